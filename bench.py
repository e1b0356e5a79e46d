#!/usr/bin/env python3
"""Benchmark of one DSA decode layer (indexer -> exact top-2048 -> sparse MLA).

Prints ONE JSON line.  A step is one pass of the whole layer (query prep,
indexer scan, top-k, sparse absorbed-MLA attention, LSE combine; plus the
shared-indexer layer where the workload has one) over one batch of synthetic
decode queries, with the caches resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload paged]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

metric: decode queries/s per layer (whole job over all ranks); the dominant
kernel's HBM roofline fraction is reported beside it.  Under torchrun (N > 1)
every rank runs its own full copy of the workload (independent sequences, no
data-path collective): weak scaling.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dsa_sparse_mla_query_gb300 import inputs as I  # noqa: E402

METRIC = "decode queries/s per layer (indexer+top-k+sparse MLA)"
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e, nominal
NOMINAL_BF16_TFLOPS = 2250.0  # dense bf16, nominal
UNIT = "queries/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="paged", choices=sorted(I.WORKLOADS) + ["insert"],
                    help="a decode layer workload, or 'insert': the cache-write side")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-s", type=float, default=1.0, help="untimed load before the timed region (clocks)")
    ap.add_argument("--seqs", type=int, default=0, help="override the number of sequences (small profiling cases)")
    ap.add_argument("--dcp", type=int, default=0,
                    help="run the layer sharded by token over this many ranks on one GPU (DCP calls)")
    ap.add_argument("--dcp-interleave", type=int, default=0,
                    help="tokens per turn of the DCP ownership (default: the page size, else 1)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws: int):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    """The largest of every rank's x (the slowest rank's time)."""
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, ws: int, ms_per_step: float) -> float:
    """Units all ranks processed per second, each rank a full copy of the
    workload (weak scaling), timed by the slowest rank."""
    return ws * units_per_rank / (ms_per_step / 1000.0)


# ---------------------------------------------------------------------------
# algorithmic bytes per launch and per step: each byte a kernel must move at least once
def index_row_bytes(wl):
    return 132 if wl.index_fp8 else 72 if wl.index_nvfp4 else 256


def latent_row_bytes(wl):
    return 656 if wl.latent_fp8 else 324 if wl.latent_nvfp4 else 1152


def dtype_name(wl) -> str:
    """The tensor-core input types the path computes in (fp32 accumulation):
    the indexer's, then the attention's when they differ.  e4m3 keys run as
    e4m3; NVFP4 keys and fp8 / NVFP4 latent rows are decoded exactly to f16."""
    idx = "e4m3" if wl.index_fp8 else "f16" if wl.index_nvfp4 else "bf16"
    att = "f16" if (wl.latent_fp8 or wl.latent_nvfp4) else "bf16"
    return idx if idx == att else f"{idx}/{att}"


def algorithmic_bytes(wl, lay):
    ctx = lay.ctx_len
    Q = wl.num_queries
    keys = sum(ctx) * index_row_bytes(wl)
    # block selection in 32-key groups: the indexer writes one maximum per group
    per_key = 4 / 32 if wl.select_block and wl.select_block % 32 == 0 else 4
    scores = int(sum(lay.ctx_len[b] for b in lay.q_seq) * per_key)
    qside = Q * (32 * 128 * 2 + 32 * 4)
    indexer = keys + scores + qside
    sel = sum(min(p + 1, wl.topk) for p in lay.q_pos)
    layers = 2 if wl.shared_layer else 1
    gather = sel * latent_row_bytes(wl) * layers
    mla_small = layers * Q * (64 * 576 * 2 + 64 * 512 * 2 + 64 * 4) + Q * wl.topk * 4
    return dict(indexer=indexer, gather=gather, step=keys + qside + gather + mla_small)


def indexer_flops(lay):
    """q.k over 128 dims for 32 heads, per causal (query, key) pair: 2 * 32 * 128 flop."""
    return sum(p + 1 for p in lay.q_pos) * 2 * 32 * 128


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        mhz, max_mhz, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1 + 0.1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                mhz.append(float(f[2]))
                max_mhz = float(f[3])
            except ValueError:
                continue
            for n, v in zip(names, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": max_mhz, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max_mhz, "reasons": sorted(reasons),
                "samples": len(mhz)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """dense bf16 (= f16) TFLOP/s, the sustained figure: the indexer is timed inside a long step"""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["bf16_tflops_sustained"]), "measured sustained bf16"
    return 1700.0, "fallback sustained bf16"


def indexer_traffic(wl_name: str, alg_bytes: int):
    """dram bytes per launch of the indexer kernel from the committed ncu
    summary, if the kernel sources still hash the same; else None.  The
    summary holds full-size launches; a launch of another size (fewer
    sequences) scales by its algorithmic bytes, as the captures themselves
    were scaled (traffic grows with the keys scanned)."""
    p = os.path.join(ROOT, "profiles", "indexer_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    if j.get("source_sha256") != kernel_source_hash() or wl_name not in j.get("per_launch_bytes", {}):
        return None
    full = j.get("algorithmic_bytes_per_launch", {}).get(wl_name)
    if not full:
        return None
    return int(round(j["per_launch_bytes"][wl_name] * alg_bytes / full))


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("indexer.cu", "indexer_nvfp4.cu", "indexer_common.cuh", "dsa_internal.cuh", "tc_ptx.cuh"):
        with open(os.path.join(ROOT, "dsa_sparse_mla_query_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
def oracle_sample(wl, n_queries: int):
    """Per sampled query: host inputs for the oracle, generated on the CPU by
    the seeded generator (same values as the device copy).  The latent rows
    are generated for the oracle's own selection only."""
    import numpy as np
    import oracle
    lay = I.make_layout(wl)
    s, b, inv = I.params(wl)
    Q = wl.num_queries
    picks = [int(x) for x in np.linspace(0, Q - 1, n_queries)]
    jobs = []
    for t in picks:
        bq = lay.q_seq[t]
        rows = lay.phys_rows(bq)
        cache = I.make_cache_rows(wl, rows, "cpu", which="index")
        q = I.make_queries(wl, "cpu", t, 1)
        jobs.append(dict(t=t, pos=lay.q_pos[t], ctx=lay.ctx_len[bq], rows=rows, keys=cache["k_idx"],
                         k_scale=cache.get("k_scale"), k_bscale=cache.get("k_bscale"), q=q, s=s, b=b, inv=inv))
    # the latent rows the oracle will select: run its indexer once here
    for j in jobs:
        j["olay"] = oracle.Layout(np.array([j["ctx"]], np.int32), j["ctx"], seq_base=np.zeros(1, np.int64))
        sc = oracle_scores(j)
        sel, m = select(wl, sc[:j["pos"] + 1])
        j["lat"] = I.make_cache_rows(wl, j["rows"][torch.from_numpy(sel[:m].astype(np.int64))], "cpu",
                                     which="latent")
        j["m"] = m
    return jobs


def oracle_scores(job):
    """The oracle's indexer scores of one sampled query over its context."""
    import numpy as np
    import oracle
    q, pos = job["q"], np.array([job["pos"]], np.int32)
    if job["k_bscale"] is not None:  # NVFP4 keys
        return oracle.index_scores_nvfp4(q["q_idx"], q["w"], job["s"], job["b"], job["inv"], np.zeros(1, np.int32),
                                         pos, job["keys"], job["k_bscale"], I.NVFP4_GLOBAL, job["olay"])[0]
    return oracle.index_scores(q["q_idx"], q["w"], job["s"], job["b"], job["inv"], np.zeros(1, np.int32), pos,
                               job["keys"], job["olay"], key_scale=job["k_scale"])[0]


def oracle_attention(wl, q, lat, m: int, which: str = "latent"):
    import numpy as np
    import oracle
    mlay = oracle.Layout(np.array([m], np.int32), m, seq_base=np.zeros(1, np.int64))
    sel = np.arange(m, dtype=np.int32)
    if wl.latent_nvfp4:
        return oracle.sparse_mla_nvfp4(q, lat[which], lat["lat_bscale"], I.NVFP4_GLOBAL, mlay, 0, sel, m,
                                       1.0 / math.sqrt(192.0))
    return oracle.sparse_mla(q, lat[which], mlay, 0, sel, m, 1.0 / math.sqrt(192.0), fp8=wl.latent_fp8)


def select(wl, causal_scores):
    """The oracle's selection: exact top-k, or blocks in block-sparse mode."""
    import oracle
    if wl.select_block:
        return oracle.block_topk(causal_scores, wl.select_block, wl.topk // wl.select_block)
    return oracle.topk(causal_scores, wl.topk)


def oracle_run(wl, job):
    """The oracle's whole layer for one query (indexer, top-k, attention)."""
    import numpy as np
    import oracle
    sc = oracle_scores(job)
    sel, m = select(wl, sc[:job["pos"] + 1])
    m = job["m"]
    oracle_attention(wl, job["q"]["q_mla"][0], job["lat"], m)
    if wl.shared_layer:
        oracle_attention(wl, job["q"]["q_mla2"][0], job["lat"], m, "latent2")


def oracle_timed(wl, jobs, threads: int) -> float:
    from concurrent.futures import ThreadPoolExecutor
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda j: oracle_run(wl, j), jobs))
    return time.perf_counter() - t0


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, wl, ws, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = cpu_threads()
    jobs = oracle_sample(wl, threads)
    for _ in range(max(args.warmup, 0)):
        oracle_timed(wl, jobs[:1], 1)
    times = [oracle_timed(wl, jobs, threads) for _ in range(args.steps)]
    total = sum(times)
    value = len(jobs) * args.steps / total
    sample = (f"{len(jobs)} queries per step (one per host thread), each the whole layer for one query of "
              f"{wl.name}: indexer over its full causal context, top-{wl.topk}, attention")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.describe(), "queries_per_step": len(jobs)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def run_ours(args, wl, ws, rank, local):
    from dsa_sparse_mla_query_gb300.runner import DecodeStep
    import dsa_sparse_mla_query_gb300 as dsa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.load()
    d = I.make_inputs(wl, dev)
    lay = d["layout"]
    step = DecodeStep(d, wl.queries_per_seq, wl.topk, device=dev, select_block=wl.select_block)
    stream = torch.cuda.current_stream(dev)
    K, W = args.steps, args.warmup
    # Two query sets alternate between steps, so consecutive steps select
    # different rows: the rows one step gathers are not in L2 for the next
    # (two gather sets, each larger than or comparable to L2, with the whole
    # index-key stream read in between).
    qsets = [None, I.make_queries(dataclasses.replace(wl, seed=wl.seed + 1), dev)]

    def events(n):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in ev:
            e.record(stream)  # creates the underlying CUDA event
        return ev

    ev = [events(4) for _ in range(K)]
    ev2 = [events(4) for _ in range(K)] if step.shared else [None] * K
    for i in range(W):
        step.run(stream, queries=qsets[i % 2])
    torch.cuda.synchronize(dev)
    if step.device_status() != 0:
        raise RuntimeError(f"device status {step.device_status()} after warm-up")

    sampler = ClockSampler(local)
    t_soak = time.time()
    t_end_soak = t_soak + args.soak_s
    while time.time() < t_end_soak:  # untimed load, so the clock samples see the timed region's state
        for i in range(20):
            step.run(stream, queries=qsets[i % 2])
        torch.cuda.synchronize(dev)
    barrier(ws)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        step.run(stream, queries=qsets[i % 2])
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ms = start.elapsed_time(end)
    # Per-stage times: a second pass of K steps with events between the stages.
    # An event between two kernels costs their programmatic overlap, so the
    # step time above comes from the pass without them.
    torch.cuda.synchronize(dev)
    for i in range(K):
        step.run(stream, events=ev[i], events2=ev2[i], queries=qsets[i % 2])
    torch.cuda.synchronize(dev)
    barrier(ws)
    t_done = time.time()
    clocks = sampler.stop(t_soak, t_done)
    ms = max_over_ranks(ms, ws, dev)
    ms_step = ms / K
    value = whole_job_rate(wl.num_queries, ws, ms_step)

    stage = lambda i, a, b: ev[i][a].elapsed_time(ev[i][b])  # noqa: E731
    idx_ms = statistics.mean(stage(i, 0, 1) for i in range(K))
    topk_ms = statistics.mean(stage(i, 1, 2) for i in range(K))
    mla_ms = statistics.mean(stage(i, 2, 3) for i in range(K))
    mla2_ms = statistics.mean(ev2[i][2].elapsed_time(ev2[i][3]) for i in range(K)) if step.shared else 0.0

    ab = algorithmic_bytes(wl, lay)
    peak, peak_kind = measured_peaks()
    achieved = ab["indexer"] / (idx_ms / 1000.0) / 1e9
    traffic = indexer_traffic(wl.name, ab["indexer"])
    # The indexer's bound: its bytes at the copy bandwidth or its q.k flops at
    # the tensor peak, whichever takes longer (the prefill chunk's 4096 queries
    # share every key, which makes it a dense contraction).
    flops = indexer_flops(lay)
    tpeak, tpeak_kind = measured_tensor_peak()
    tensor_bound = flops / (tpeak * 1e12) > ab["indexer"] / (peak * 1e9)

    # ---- end to end through the C ABI with host buffers, as a serving loop
    # runs it: every step's query inputs come from pinned host memory and its
    # outputs go back to pinned host memory, on their own streams, so that the
    # next step's inputs and the last step's outputs move while a step
    # computes.  Two sets of device inputs, outputs and workspace alternate;
    # events keep a set's inputs from being overwritten before its previous
    # step has computed, and its outputs before they have been read back.
    keys = ["q_idx", "w", "q_mla"] + (["q_mla2"] if step.shared else [])
    host_in = {k: d[k].cpu().pin_memory() for k in keys}
    host_pos = d["q_pos"].cpu().pin_memory()
    d_b = dict(d, **{k: torch.empty_like(d[k]) for k in keys + ["q_pos"]})
    for k in keys + ["q_pos"]:
        d_b[k].copy_(d[k])
    step_b = DecodeStep(d_b, wl.queries_per_seq, wl.topk, device=dev, select_block=wl.select_block)
    sets = [(step, d), (step_b, d_b)]

    def outs_of(st):
        return [st.out, st.lse, st.idx, st.topk_len] + ([st.out2, st.lse2] if st.shared else [])
    host_out = [[o.cpu().pin_memory() for o in outs_of(st)] for st, _ in sets]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values()) + host_pos.numel() * 4
    d2h = sum(o.numel() * o.element_size() for o in host_out[0])
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    Ke = max(2, K)
    barrier(ws)
    torch.cuda.synchronize(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ready, done, read = [ev() for _ in range(Ke)], [ev() for _ in range(Ke)], [ev() for _ in range(Ke)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(Ke):
        st, dd = sets[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(done[i - 2])  # this set's previous step has computed
            for k, v in host_in.items():
                dd[k].copy_(v, non_blocking=True)
            dd["q_pos"].copy_(host_pos, non_blocking=True)
            ready[i].record(s_in)
        stream.wait_event(ready[i])
        if i >= 2:
            stream.wait_event(read[i - 2])  # this set's previous outputs are back on the host
        st.run(stream)
        done[i].record(stream)
        s_out.wait_event(done[i])
        with torch.cuda.stream(s_out):
            for o, h in zip(outs_of(st), host_out[i % 2]):
                h.copy_(o, non_blocking=True)
            read[i].record(s_out)
    stream.wait_event(read[Ke - 1])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e2e_ms = e0.elapsed_time(e1) / Ke
    e2e_ms = max_over_ranks(e2e_ms, ws, dev)
    if step.device_status() != 0 or step_b.device_status() != 0:
        raise RuntimeError(f"device status {step.device_status()} / {step_b.device_status()}")

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = cpu_threads()
        jobs = oracle_sample(wl, 6 * threads)
        secs = oracle_timed(wl, jobs, threads)
        cpu = {"value": len(jobs) / secs, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{len(jobs)} queries of {wl.name} spread over the batch, each the whole layer "
                         f"(indexer over the full causal context, top-{wl.topk}, attention), "
                         f"{threads} threads of the single-threaded fp64 oracle, {secs:.1f} s wall"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": dtype_name(wl), "data": "synthetic",
            "config": {"workload": wl.describe(), "queries": wl.num_queries, "global_batch": ws * wl.num_queries,
                       "l2": "inputs larger than L2 (index keys %.0f MB read every step, latent cache %.0f MB); "
                             "two query sets alternate between steps, so consecutive steps gather different "
                             "rows (%.0f MB each)"
                             % (sum(lay.ctx_len) * index_row_bytes(wl) / 1e6,
                                lay.num_rows * latent_row_bytes(wl) / 1e6, ab["gather"] / 1e6),
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "roofline": ({"bound": "tensor", "achieved": flops / (idx_ms / 1000.0) / 1e12, "peak": tpeak,
                          "unit": "TFLOP/s", "frac": flops / (idx_ms / 1000.0) / 1e12 / tpeak, "traffic": traffic,
                          "kernel": "indexer (query prep + key scan)", "algorithmic_flops_per_launch": flops,
                          "algorithmic_bytes_per_launch": ab["indexer"], "ms_per_launch": idx_ms,
                          "peak_kind": tpeak_kind,
                          "frac_of_nominal": flops / (idx_ms / 1000.0) / 1e12 / NOMINAL_BF16_TFLOPS,
                          "note": "flops of q.k over 128 dims; the kernel's MMAs do %.1fx that%s"
                                  % ((1.5, " (rotated dims in hi + lo)") if wl.rope else (1.0, ""))}
                         if tensor_bound else
                         {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                          "frac": achieved / peak, "traffic": traffic, "kernel": "indexer (query prep + key scan)",
                          "algorithmic_bytes_per_launch": ab["indexer"], "ms_per_launch": idx_ms,
                          "peak_kind": f"{peak_kind} HBM copy", "frac_of_nominal": achieved / NOMINAL_HBM_GBS}),
            "layer": {"algorithmic_bytes_per_step": ab["step"],
                      "achieved_gbs": ab["step"] / (ms_step / 1000.0) / 1e9,
                      "frac_of_peak": ab["step"] / (ms_step / 1000.0) / 1e9 / peak,
                      "stage_ms": {"indexer": idx_ms, "topk": topk_ms, "mla": mla_ms, "mla_shared_layer": mla2_ms},
                      "stage_timing": "second pass of the same K steps with CUDA events between the stages",
                      "keys_scanned_per_s": ws * sum(lay.ctx_len) / (ms_step / 1000.0)},
            "e2e": {"value": whole_job_rate(wl.num_queries, ws, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "how": "each step's query inputs copied from pinned host memory and its outputs to pinned host "
                           "memory on their own streams, two buffer sets alternating (copies overlap other steps' "
                           "compute)"},
            "gpu_launches": K * step.launches_per_step(),  # kernels of the timed pass
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_dcp(args, wl, ws, rank, local):
    """The layer sharded by token over args.dcp ranks whose shards share this
    GPU: per rank the indexer and its top-k candidates, the selector's merge,
    per rank compaction and attention, the LSE combine (dcp.ShardedLayer)."""
    from dsa_sparse_mla_query_gb300.dcp import ShardedLayer
    import dsa_sparse_mla_query_gb300 as dsa
    from dsa_sparse_mla_query_gb300 import _binding as B

    R = args.dcp
    inter = args.dcp_interleave or (wl.page_size or 1)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = cpu_threads()
        jobs = oracle_sample(wl, 6 * threads)
        secs = oracle_timed(wl, jobs, threads)
        cpu = {"value": len(jobs) / secs, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{len(jobs)} queries of {wl.name}, each the whole (unsharded) layer, "
                         f"{threads} threads of the fp64 oracle, {secs:.1f} s wall"}
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.load()
    d = I.make_inputs(wl, dev)
    lay = d["layout"]
    sh = ShardedLayer(d, wl.queries_per_seq, wl.topk, R, inter, device=dev)
    stream = torch.cuda.current_stream(dev)
    K, W = args.steps, args.warmup

    def phase_ok(name):  # outside the timed regions
        torch.cuda.synchronize(dev)
        if sh.device_status() != 0:
            raise RuntimeError(f"device status {sh.device_status()} after {name}")

    for _ in range(W):
        sh.run(stream)
    phase_ok("warm-up")
    sampler = ClockSampler(local)
    t_soak = time.time()
    while time.time() < t_soak + args.soak_s:
        for _ in range(20):
            sh.run(stream)
        torch.cuda.synchronize(dev)
    phase_ok("the untimed load")
    barrier(ws)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(K):
        sh.run(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    ms_step = max_over_ranks(start.elapsed_time(end) / K, ws, dev)
    phase_ok("the timed steps")
    # stages: a second pass with events between them
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    for i in range(K):
        sh.run(stream, marks=marks[i])
    phase_ok("the stage-timing steps")
    st = lambda a, b: statistics.mean(m[a].elapsed_time(m[b]) for m in marks)  # noqa: E731
    stages = {"indexers_and_candidates": st(0, 1), "merge": st(1, 2), "compact_and_attention": st(2, 3),
              "lse_combine": st(3, 4)}
    # the indexer of every rank alone, events around each launch
    kd = B.DSA_FP8_E4M3_ROWSCALE if sh.k_fp8 else B.DSA_BF16
    iev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * R)] for _ in range(K)]
    for i in range(K):
        for r, v in enumerate(sh.views):
            iev[i][2 * r].record(stream)
            B.dsa_index_scores(d["q_idx"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], v.k_idx, v.k_scale, kd,
                               v.seqs, sh.num_q, v.scores, v.ld, sh.ws, sh.ws_bytes, sh.status, stream)
            iev[i][2 * r + 1].record(stream)
    phase_ok("the indexer-timing pass")
    t_done = time.time()
    clocks = sampler.stop(t_soak, t_done)
    idx_ms = statistics.mean(sum(e[2 * r].elapsed_time(e[2 * r + 1]) for r in range(R)) for e in iev)
    # end to end: the step's query inputs from pinned host memory, outputs back
    keys = ["q_idx", "w", "q_mla"] + (["q_mla2"] if sh.shared else [])
    host_in = {k: d[k].cpu().pin_memory() for k in keys}
    host_pos = d["q_pos"].cpu().pin_memory()
    outs = [sh.out, sh.lse, sh.idx, sh.topk_len] + ([sh.out2, sh.lse2] if sh.shared else [])
    host_out = [o.cpu().pin_memory() for o in outs]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values()) + host_pos.numel() * 4
    d2h = sum(o.numel() * o.element_size() for o in host_out)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        for k, v in host_in.items():
            d[k].copy_(v, non_blocking=True)
        d["q_pos"].copy_(host_pos, non_blocking=True)
        sh.run(stream)
        for o, h in zip(outs, host_out):
            h.copy_(o, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, ws, dev)
    phase_ok("the end-to-end steps")
    ab = algorithmic_bytes(wl, lay)
    peak, peak_kind = measured_peaks()
    achieved = ab["indexer"] / (idx_ms / 1000.0) / 1e9
    lat = B.DSA_FP8_DS_MLA if sh.lat_fp8 else B.DSA_BF16
    per_rank = [B.dsa_decode_layer_launches(v.seqs, sh.num_q, wl.topk, 0, lat) + 2 +
                (B.dsa_decode_layer_launches(v.seqs, sh.num_q, wl.topk, 1, lat) if sh.shared else 0)
                for v in sh.views]
    launches = sum(per_rank) + 1 + (2 if sh.shared else 1)
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": whole_job_rate(wl.num_queries, ws, ms_step), "unit": UNIT, "n_gpus": ws,
            "steps": K, "warmup": W, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype_name(wl), "data": "synthetic",
            "config": {"workload": wl.describe(), "queries": wl.num_queries,
                       "dcp": f"sharded by token over {R} ranks in turns of {inter} tokens, every shard on this GPU",
                       "l2": "inputs larger than L2",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": None, "kernel": f"indexer over the {R} shards (query prep + key scan per rank)",
                         "algorithmic_bytes_per_launch": ab["indexer"], "ms_per_launch": idx_ms,
                         "peak_kind": f"{peak_kind} HBM copy", "frac_of_nominal": achieved / NOMINAL_HBM_GBS},
            "stages_ms": stages,
            "e2e": {"value": whole_job_rate(wl.num_queries, ws, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": K * launches, "clocks": clocks, "cpu_baseline": cpu}), flush=True)


INSERT_TOKENS = 1 << 20
INSERT_KEY_BYTES = 256 + 132 + 8 + 4        # x in; e4m3 row + scale out; slot + position
INSERT_LATENT_BYTES = 1024 + 128 + 656 + 8 + 4  # c_kv + k_pe in; fp8_ds_mla row out; slot + position
INSERT_BYTES_PER_TOKEN = INSERT_KEY_BYTES + INSERT_LATENT_BYTES
INSERT_ORACLE_TOKENS = 1024


def insert_oracle_step(h) -> None:
    """The oracle's cache-write step: key rows and latent rows with their e4m3 codes."""
    import oracle
    k = oracle.index_k(h["x"], h["gamma"], h["beta"], 1e-6, h["pos"], h["inv_freq"])
    oracle.quantize_rows_e4m3(k, 128)
    lat = oracle.latent_k(h["c_kv"], h["k_pe"], h["pos"], h["inv_freq"])
    oracle.quantize_rows_e4m3(lat[:, :512], 128)


def insert_oracle_inputs():
    import oracle
    oracle.build()
    return I.make_insert_inputs(INSERT_ORACLE_TOKENS, 1, INSERT_ORACLE_TOKENS, "cpu", seed=0, page_size=64)


INSERT_SAMPLE = (f"{INSERT_ORACLE_TOKENS} new tokens per step (key and latent rows with their e4m3 codes), "
                 "one host thread")


def run_insert(args, ws, rank, local):
    """The cache-write side: a step inserts INSERT_TOKENS new tokens (indexer
    key: LayerNorm + RoPE + e4m3 with a row scale; latent: RoPE + fp8_ds_mla)
    into caches of as many rows, 64-token pages in a random order.  HBM-bound:
    2,220 algorithmic bytes per token, 1,820 of them the latent insert's."""
    n = INSERT_TOKENS
    metric, unit = "cache-insert tokens/s (indexer key e4m3 + fp8_ds_mla latent)", "tokens/s"
    cfg = {"workload": f"insert: {n} new tokens, LayerNorm + RoPE + e4m3/row-scale indexer keys and RoPE + "
                       f"fp8_ds_mla latent rows into {n}-row caches of 64-token pages in a random page order",
           "l2": "inputs larger than L2 (%.0f MB in, %.0f MB out per step)" % (n * 1432 / 1e6, n * 788 / 1e6),
           "parallelism": "single GPU" if ws == 1 else f"replicas x{ws}"}
    if args.impl == "reference":
        h = insert_oracle_inputs()
        K = max(1, args.steps)
        t0 = time.time()
        for _ in range(K):
            insert_oracle_step(h)
        secs = (time.time() - t0) / K
        v = INSERT_ORACLE_TOKENS / secs
        print(json.dumps({"metric": metric, "value": v, "unit": unit, "n_gpus": ws, "steps": K, "warmup": 0,
                          "ms_per_step": secs * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "f64", "data": "synthetic", "config": cfg, "impl": "reference",
                          "cpu_baseline": {"value": v, "unit": unit, "cores": 1, "kind": "oracle",
                                           "sample": INSERT_SAMPLE},
                          "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return
    import dsa_sparse_mla_query_gb300 as dsa
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        h = insert_oracle_inputs()  # before the first CUDA call
        t0 = time.time()
        for _ in range(3):
            insert_oracle_step(h)
        secs = (time.time() - t0) / 3
        cpu = {"value": INSERT_ORACLE_TOKENS / secs, "unit": unit, "cores": 1, "kind": "oracle",
               "sample": INSERT_SAMPLE + ", 3 steps"}
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.load()
    d = I.make_insert_inputs(n, 1, n, dev, seed=0, page_size=64)
    keys = torch.zeros((n, 128), dtype=torch.uint8, device=dev)
    k_scale = torch.zeros(n, dtype=torch.float32, device=dev)
    latent = torch.zeros((n, I.DS_MLA_ROW_BYTES), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def key_insert():
        dsa.dsa_index_k_insert(d["x"], d["gamma"], d["beta"], 1e-6, d["pos"], d["inv_freq"], d["slot"], n, keys,
                               k_scale, dsa.DSA_FP8_E4M3_ROWSCALE, n, st, stream)

    def latent_insert():
        dsa.dsa_latent_insert(d["c_kv"], d["k_pe"], d["pos"], d["inv_freq"], d["slot"], n, latent,
                              dsa.DSA_FP8_DS_MLA, n, st, stream)

    def step():
        key_insert()
        latent_insert()

    K, W = args.steps, args.warmup
    for _ in range(W):
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local)
    t_soak = time.time()
    while time.time() < t_soak + args.soak_s:
        for _ in range(20):
            step()
        torch.cuda.synchronize(dev)
    barrier(ws)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    t_done = time.time()
    ms = max_over_ranks(e0.elapsed_time(e1) / K, ws, dev)
    clocks = sampler.stop(t_soak, t_done)
    # each kernel alone, events on its stream around each launch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        ev[i][0].record(stream)
        key_insert()
        ev[i][1].record(stream)
        latent_insert()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    key_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    lat_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    # end to end: the new tokens' inputs from pinned host memory each step, the status word back
    keys_in = ["x", "c_kv", "k_pe", "pos", "slot"]
    host = {k: d[k].cpu().pin_memory() for k in keys_in}
    st_h = torch.zeros(1, dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    e0.record(stream)
    for _ in range(K):
        for k, v in host.items():
            d[k].copy_(v, non_blocking=True)
        step()
        st_h.copy_(st, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, ws, dev)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    peak, peak_kind = measured_peaks()
    lat_bytes = n * INSERT_LATENT_BYTES
    achieved = lat_bytes / (lat_ms / 1000.0) / 1e9
    step_gbs = n * INSERT_BYTES_PER_TOKEN / (ms / 1000.0) / 1e9
    if rank != 0:
        return
    print(json.dumps({"metric": metric, "value": whole_job_rate(n, ws, ms), "unit": unit, "n_gpus": ws, "steps": K,
                      "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                      "vs_baseline": None, "dtype": "e4m3/bf16", "data": "synthetic", "config": cfg,
                      "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                                   "frac": achieved / peak, "traffic": None, "kernel": "latent_insert_kernel<fp8>",
                                   "algorithmic_bytes_per_launch": lat_bytes, "peak_kind": f"{peak_kind} HBM copy",
                                   "frac_of_nominal": achieved / NOMINAL_HBM_GBS},
                      "stages_ms": {"index_k_insert": key_ms, "latent_insert": lat_ms},
                      "step_hbm": {"achieved": step_gbs, "frac": step_gbs / peak,
                                   "bytes": n * INSERT_BYTES_PER_TOKEN},
                      "e2e": {"value": whole_job_rate(n, ws, e2e_ms), "unit": unit, "h2d_bytes_per_step": h2d,
                              "d2h_bytes_per_step": 4},
                      "gpu_launches": 2 * K, "clocks": clocks, "cpu_baseline": cpu}))


def main():
    args = parse()
    ws, rank, local = dist_env()
    wl = None
    if args.workload != "insert":
        wl = I.WORKLOADS[args.workload]
        if args.seqs:
            wl = I.scaled(wl, num_seqs=args.seqs)
        if args.dcp and (wl.index_nvfp4 or wl.latent_nvfp4):
            raise SystemExit("--dcp shards bf16 and e4m3 caches; the NVFP4 workloads run unsharded")
    if args.impl == "reference":
        # the oracle on the host cores: rank 0 alone runs and prints
        if ws > 1 and rank != 0:
            return
        if wl is None:
            run_insert(args, ws, rank, local)
        else:
            run_reference(args, wl, ws, rank)
        return
    if ws > 1:
        torch.distributed.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    try:
        if wl is None:
            run_insert(args, ws, rank, local)
        elif args.dcp:
            run_dcp(args, wl, ws, rank, local)
        else:
            run_ours(args, wl, ws, rank, local)
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
