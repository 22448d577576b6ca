#!/usr/bin/env python3
"""Benchmark: decode layer-steps/s of top-k sparse attention over a two-level
KV cache, on the batch-16 / 4-layer / 32K-context workload by default.

One step = one decode step of every request over every layer: for each layer,
append the new token (index key to HBM, K/V row to the pinned host copy) and
run hs_decode_layer (indexer + top-k, RESOLVE, attention).  value = layer-steps
per second (one layer-step = one layer of all R requests); tokens/s = R * steps
per second.  The timed steps are captured once into a CUDA graph and replayed,
as a serving engine's decode graph would be; every kernel still runs every
step.  e2e repeats the measurement through the Python API with the step's
inputs copied host -> device and the outputs device -> host inside the loop.

--impl reference times the CPU oracle on the same workload (a bounded sample
of requests per step, scaled to the whole batch).
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
sys.path.insert(0, ROOT)

import workload as wl  # noqa: E402

METRIC = "sparse-decode layer-steps/s"
UNIT = "layer-steps/s"
L2_BYTES = 129 * 2 ** 20


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_workload(w: wl.Workload, rank: int, world: int) -> wl.Workload:
    """Weak scaling: each rank serves its own batch of requests (its own seed)."""
    if world <= 1:
        return w
    import dataclasses
    return dataclasses.replace(w, seed=w.base_seed + 1000 * rank)


def max_over_ranks(x: float, world: int) -> float:
    """Slowest rank's time (torch.distributed, timing only: no data-path collective)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_tflops():
    """Sustained dense bf16 tensor throughput (the kernels run inside a long step)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured (sustained)"
    return 1700.0, "fallback (sustained)"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 10):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []

    def start(self):
        if self.interval_ms <= 0:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, window=None) -> dict:
        """Summary of the samples taken inside window = (t0, t1) (wall time), or of
        all samples when none fell inside it."""
        if self.proc is None:
            why = "not sampled (--clock-interval-ms 0)" if self.interval_ms <= 0 else "nvidia-smi unavailable"
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [why]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = [ln for t, ln in self.lines if window and window[0] <= t <= window[1]]
        for ln in inside or [ln for _, ln in self.lines]:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "timed region" if inside else "whole run (no sample fell inside the timed region)"}


def code_hash(path: str) -> str:
    """First 16 hex digits of the SHA-256 of a source file's code lines: line
    comments and blank lines are dropped, so an edit of comments alone keeps the
    hash (and the ncu figures taken on that code)."""
    code = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.split("//", 1)[0].strip()
            if line:
                code.append(line)
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


def kernel_source_hash(name: str) -> str:
    return code_hash(os.path.join(ROOT, "tiered_kv_cache_int8_gb300", "csrc", name))


KERNEL_FILES = {"append": "hs_append.cu", "select": "hs_select.cu", "attention": "hs_attention.cu"}


def host_store_pages(stats: dict) -> dict:
    """How much of the pinned host K/V store is backed by transparent huge pages
    (the library faults it in and collapses what the kernel backed with base
    pages; random row reads over the link take about half as long on huge
    pages), from hs_stats; plus the system's THP mode (read only)."""
    out = {"thp_frac": round(stats["host_huge_bytes"] / max(1, stats["host_bytes"]), 4)}
    for name in ("enabled", "defrag"):
        try:
            with open(f"/sys/kernel/mm/transparent_hugepage/{name}") as f:
                out[f"thp_{name}"] = f.read().strip()
        except OSError:
            out[f"thp_{name}"] = None
    return out


def ncu_traffic(kernel: str, workload: str, latent: bool = False):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this kernel source and workload (else None).  Latent-row attention lives in
    its own source file."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    src = "hs_attention_mla.cu" if (latent and kernel == "attention") else KERNEL_FILES[kernel]
    if not e or e.get("source_sha") != kernel_source_hash(src):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# algorithmic traffic of one layer of all R requests (per kernel)
# ---------------------------------------------------------------------------

def algorithmic_bytes(w: wl.Workload, n_ctx: np.ndarray, misses: float, resolve_pulls: bool = False,
                      selects: bool = True, page_size: int = 1) -> dict:
    """HBM and host-link bytes the method itself moves for one layer-step of all
    requests, per kernel.  n_ctx: context length of each request at this step;
    misses: rows pulled from host memory in this layer-step (all requests);
    resolve_pulls: the missed rows are copied (host read, slot write) by RESOLVE
    inside the select kernel rather than by the attention kernel.

    select: the index-key scan and query (the indexer), then per request the
    selection, slot and page-table reads/writes (16 B per selected position), the
    stamp/reverse scan (8 B per slot), 12 B of metadata per miss, and the appended
    token (its row read from HBM and written to the host copy, its key).
    attention: every selected row, its slot, the queries and the outputs.
    selects=False: a layer that reuses its group lead's selection (index sharing)
    scans no index keys; its selection, slot and metadata bytes still move (the
    lead's call writes them for it).
    page_size P > 1 (page selection): the scan reads each page's bounds (2 d_idx
    bytes per page) instead of every key, slot metadata is per page slot (B / P),
    and the appended token also updates its page's bounds; misses count rows."""
    k_eff = np.minimum(w.top_k, n_ctx)
    R = w.n_requests
    row = w.row_bytes
    P = max(1, int(page_size))
    scan = (n_ctx * w.d_idx).sum() if P == 1 else (((n_ctx + P - 1) // P) * 2 * w.d_idx).sum()
    hbm = {
        "append": 0.0,
        "select": (float(scan) + R * w.d_idx if selects else 0.0)
        + float(k_eff.sum()) * (4 + 4 + 4 + 4) + R * (w.hot_slots // P) * 8 + misses / P * 12
        + R * (w.row_bytes + 2 * w.d_idx + 4) + (R * 4 * w.d_idx if P > 1 else 0),
        "attention": float(k_eff.sum()) * (row + 4) + R * w.h_q * (w.d_qk + w.d_v) * 2,
    }
    link = {"append": 0.0, "select": R * row, "attention": 0.0}
    puller = "select" if resolve_pulls else "attention"
    hbm[puller] += misses * row    # the slot writes
    link[puller] += misses * row   # the host reads
    return {"hbm": hbm, "link": link}


def resolve_pulls(fetch_mode: int, shared_kv: bool) -> bool:
    """Which kernel copies the missed rows: RESOLVE (in the select kernel) for
    fetch mode 1 and for latent rows, else the attention kernel's loader."""
    return shared_kv or fetch_mode == 1


def attention_timeline(st0: dict, st1: dict, n_launch: int, n_cta: int):
    """Host-link exposure and load balance of the GQA attention kernel between two
    hs_stats snapshots (None for latent rows, which record nothing).  A consumer
    warp per CTA times its wait for every stage of rows; a stage holding a row read
    from host memory waits longer than one of HBM rows only, and that excess, summed
    over a CTA's host stages, is the link time the CTA could not hide."""
    d = {k: st1[k] - st0[k] for k in ("att_host_wait_ns", "att_host_stages", "att_hbm_wait_ns", "att_hbm_stages")}
    if d["att_host_stages"] + d["att_hbm_stages"] == 0 or n_launch == 0:
        return None
    hbm_mean = d["att_hbm_wait_ns"] / max(1, d["att_hbm_stages"])
    host_mean = d["att_host_wait_ns"] / max(1, d["att_host_stages"])
    exposed = max(0.0, d["att_host_wait_ns"] - d["att_host_stages"] * hbm_mean)
    span, med = st1["att_last_span_ns"], st1["att_last_median_ns"]
    return {"host_stage_wait_us": round(host_mean / 1e3, 3), "hbm_stage_wait_us": round(hbm_mean / 1e3, 3),
            "host_stages_per_cta_layer": round(d["att_host_stages"] / (n_launch * n_cta), 2),
            "link_exposed_us_per_cta_layer": round(exposed / (n_launch * n_cta) / 1e3, 3),
            "last_launch_span_us": round(span / 1e3, 2), "last_launch_median_cta_end_us": round(med / 1e3, 2),
            "span_over_median": round(span / med, 3) if med else None,
            "note": "consumer waits per stage of 16 rows, summed over CTAs; exposed = host-stage waits minus "
                    "the mean HBM-stage wait per host stage; span and median CTA end from the first CTA's start "
                    "of the timed region's last attention launch"}


def graph_upload(g, stream) -> bool:
    """Uploads an instantiated CUDA graph to the device (cudaGraphUpload) so
    that the timed replay does not pay the first launch's upload; False when the
    installed torch does not expose the executable graph."""
    import ctypes
    try:
        exe = int(g.raw_cuda_graph_exec())
        rt = ctypes.CDLL("libcudart.so.13")
    except (AttributeError, RuntimeError, OSError, TypeError):
        return False
    rt.cudaGraphUpload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    rt.cudaGraphUpload.restype = ctypes.c_int
    return rt.cudaGraphUpload(ctypes.c_void_p(exe), ctypes.c_void_p(stream.cuda_stream)) == 0


def link_peak_gbs(dev, nbytes=1 << 30, reps=5) -> float:
    """Pinned host -> device cudaMemcpyAsync bandwidth (best of reps)."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = 0.0
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize(dev)
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del src, dst
    return best


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_cache(w: wl.Workload, r: int, l: int, replacement: str):
    """The oracle's hot cache of one (request, layer) under the chosen policy
    (the random policy's seed is the library default, 0)."""
    from oracle import FIFOHotCache, LRUHotCache, RandomHotCache
    if replacement == "random":
        return RandomHotCache(w.hot_slots, seed=0, request=r, layer=l, n_layers=w.n_layers)
    return {"lru": LRUHotCache, "fifo": FIFOHotCache}[replacement](w.hot_slots)


def oracle_sample(w: wl.Workload, requests, layers, steps: int, replacement: str = "lru") -> tuple[float, int]:
    """Times the oracle over decode steps 0..steps-1 of the given (request, layer)
    pairs; returns (seconds, request-layer-steps).  Input generation is not timed."""
    from oracle import indexer_scores_many, sparse_attention, topk_select
    total = 0.0
    units = 0
    for l in layers:
        for r in requests:
            keys = wl.idx_keys_upto(w, r, l, steps)
            walk = wl.query_walk(w, r, l, steps)
            kv = wl.prefill_kv(w, r, l)
            n0 = int(w.contexts()[r])
            qs = [wl.step_query(w, r, l, t) for t in range(steps)]
            app = [wl.step_kv_row(w, r, l, t) for t in range(steps)]
            cache = oracle_cache(w, r, l, replacement)
            t0 = time.perf_counter()
            for t in range(steps):
                n = n0 + t + 1
                s = indexer_scores_many(keys[:n], walk[t])[:, 0]
                sel = topk_select(s, w.top_k)
                cache.step(sel)
                rows = np.empty((sel.size, w.row_elems), np.uint16)
                pre = sel < n0
                rows[pre] = kv[sel[pre]]
                for i in np.nonzero(~pre)[0]:
                    rows[i] = app[int(sel[i] - n0)]
                sparse_attention(qs[t], rows, h_kv=w.h_kv, d_qk=w.d_qk, d_v=w.d_v, v_offset=w.v_offset)
            total += time.perf_counter() - t0
            units += steps
    return total, units


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def policy_floor(args, w: wl.Workload, dev_index: int, n_pairs: int = 2, steps: int = 64) -> dict:
    """Misses of the configured replacement policy against Belady's MIN on the same
    GPU-selected trace (the floor the pages compare their policies with): a fresh
    cache of the first n_pairs requests of layer 0 runs `steps` decode steps from
    cold with the selections read back, outside every timed region."""
    import torch
    from tiered_kv_cache_int8_gb300 import HiSparseCache
    from tiered_kv_cache_int8_gb300.analysis import belady_misses
    dev = torch.device("cuda", dev_index)
    R = min(n_pairs, w.n_requests)
    n0 = w.contexts()[:R]
    cache = HiSparseCache(n_layers=1, max_requests=R, max_context=int(n0.max()) + steps, h_q=w.h_q, h_kv=w.h_kv,
                          d_qk=w.d_qk, d_v=w.d_v, d_idx=w.d_idx, top_k=w.top_k, hot_slots=w.hot_slots,
                          shared_kv=w.shared_kv, device=dev_index, fetch_mode=args.fetch_mode,
                          replacement=args.replacement)
    try:
        for r in range(R):
            n = int(n0[r])
            kv = torch.from_numpy(wl.prefill_kv(w, r, 0).view(np.int16)).to(dev)
            keys = torch.from_numpy(wl.prefill_idx_keys(w, r, 0)).to(dev)
            rid = torch.tensor([r], dtype=torch.int32, device=dev)
            cache.append(0, kv.view(1, n, w.row_elems), keys.view(1, n, w.d_idx), req_ids=rid)
            torch.cuda.synchronize(dev)
        walks = [wl.query_walk(w, r, 0, steps) for r in range(R)]
        sel = torch.empty((steps, R, w.top_k), dtype=torch.int32, device=dev)
        for t in range(steps):
            q_idx = torch.from_numpy(np.stack([walks[r][t] for r in range(R)])).to(dev)
            q = torch.from_numpy(np.stack([wl.step_query(w, r, 0, t) for r in range(R)]).view(np.int16)).to(dev)
            new_kv = torch.from_numpy(np.stack([wl.step_kv_row(w, r, 0, t) for r in range(R)]).view(np.int16)).to(dev)
            new_keys = torch.from_numpy(np.stack([wl.step_idx_key(w, r, 0, t) for r in range(R)])).to(dev)
            cache.decode_layer(0, q_idx, q, sel_out=sel[t], new_kv=new_kv, new_keys=new_keys)
        st = cache.stats()
        trace = sel.cpu().numpy()
    finally:
        cache.close()
    accesses = st["hits"] + st["misses"]
    floor = 0
    for r in range(R):
        floor += belady_misses([trace[t, r][trace[t, r] >= 0] for t in range(steps)], w.hot_slots)
    return {"policy": args.replacement, "requests": R, "layer": 0, "steps": steps, "from": "cold",
            "accesses": int(accesses), "misses": int(st["misses"]), "belady_misses": int(floor),
            "miss_rate": round(st["misses"] / max(1, accesses), 5),
            "belady_miss_rate": round(floor / max(1, accesses), 5)}


def run_hisparse(args, w: wl.Workload, rank: int, world: int, dev_index: int) -> dict | None:
    import torch

    from tiered_kv_cache_int8_gb300 import HiSparseCache
    from tiered_kv_cache_int8_gb300.build import build

    build()
    dev = torch.device("cuda", dev_index)
    torch.cuda.set_device(dev)
    W, K = args.warmup, args.steps
    T = W + 2 * K + args.e2e_steps
    R, L = w.n_requests, w.n_layers
    cache = HiSparseCache(n_layers=L, max_requests=R, max_context=w.max_context(T), h_q=w.h_q, h_kv=w.h_kv,
                          d_qk=w.d_qk, d_v=w.d_v, d_idx=w.d_idx, top_k=w.top_k, hot_slots=w.hot_slots,
                          shared_kv=w.shared_kv, device=dev_index, fetch_mode=args.fetch_mode,
                          replacement=args.replacement, index_share=args.index_share,
                          share_prefetch=bool(args.share_prefetch), page_size=args.page_size)

    # ---- prefill: generate each (request, layer) context and append it -----------
    t_pre = time.time()
    n0 = w.contexts()
    stage_kv = torch.empty((int(n0.max()), w.row_elems), dtype=torch.int16, pin_memory=True)
    stage_keys = torch.empty((int(n0.max()), w.d_idx), dtype=torch.int8, pin_memory=True)
    for l in range(L):
        for r in range(R):
            n = int(n0[r])
            wl.prefill_kv(w, r, l, out=stage_kv[:n].numpy().view(np.uint16))
            stage_keys[:n].numpy()[:] = wl.prefill_idx_keys(w, r, l)
            rid = torch.tensor([r], dtype=torch.int32, device=dev)
            cache.append(l, stage_kv[:n].view(1, n, w.row_elems), stage_keys[:n].view(1, n, w.d_idx), req_ids=rid)
            torch.cuda.synchronize(dev)   # the staging buffer is reused
    del stage_kv, stage_keys
    t_pre = time.time() - t_pre
    host_pages = host_store_pages(cache.stats())

    # ---- per-step inputs, resident in HBM -----------------------------------------
    walks = np.stack([np.stack([wl.query_walk(w, r, l, T) for r in range(R)]) for l in range(L)])  # [L,R,T,d]
    q_idx = torch.from_numpy(np.ascontiguousarray(walks.transpose(2, 0, 1, 3))).to(dev)             # [T,L,R,d]
    q_host = np.empty((T, L, R, w.h_q, w.d_qk), np.uint16)
    kv_host = np.empty((T, L, R, 1, w.row_elems), np.uint16)
    key_host = np.empty((T, L, R, 1, w.d_idx), np.int8)
    for t in range(T):
        for l in range(L):
            for r in range(R):
                q_host[t, l, r] = wl.step_query(w, r, l, t)
                kv_host[t, l, r, 0] = wl.step_kv_row(w, r, l, t)
                key_host[t, l, r, 0] = wl.step_idx_key(w, r, l, t)
    q_dev = torch.from_numpy(q_host.view(np.int16)).to(dev)
    kv_dev = torch.from_numpy(kv_host.view(np.int16)).to(dev)
    key_dev = torch.from_numpy(key_host).to(dev)
    out_dev = torch.empty((L, R, w.h_q, w.d_v), dtype=torch.bfloat16, device=dev)

    stream = torch.cuda.Stream(dev)

    def enqueue_step(t):
        for l in range(L):   # the new token's append rides on the decode call
            cache.decode_layer(l, q_idx[t, l], q_dev[t, l], out=out_dev[l], stream=stream,
                               new_kv=kv_dev[t, l], new_keys=key_dev[t, l])

    # ---- warm-up (eager) ------------------------------------------------------------
    with torch.cuda.stream(stream):
        for t in range(W):
            enqueue_step(t)
    torch.cuda.synchronize(dev)
    st0 = cache.stats()

    uploaded = []

    def capture(t_begin, t_end):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                for t in range(t_begin, t_end):
                    enqueue_step(t)
        uploaded.append(graph_upload(g, stream))   # the first launch's upload stays outside the timing
        torch.cuda.synchronize(dev)
        return g

    def replay_timed(g):
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(e0.elapsed_time(e1), world)

    # ---- timed region A: the K steps as one CUDA graph (the headline value) ----------
    graph = capture(W, W + K)
    clocks = ClockSampler(dev_index, args.clock_interval_ms)
    clocks.start()
    time.sleep(0.5)   # the sampler's start-up (NVML initialisation) stays out of the timed region
    t_wall0 = time.time()
    ms_total = replay_timed(graph)
    clk = clocks.stop(window=(t_wall0, time.time()))
    del graph
    st1 = cache.stats()
    misses = st1["misses"] - st0["misses"]
    hits = st1["hits"] - st0["hits"]

    # ---- timed region B: the next K steps with every kernel bracketed by events -------
    cache.set_timing(True)
    graph_b = capture(W + K, W + 2 * K)
    ms_total_b = replay_timed(graph_b)
    ktimes = cache.kernel_times()
    timing_mode = "events in the CUDA graph"
    if sum(n for _, n in ktimes.values()) == 0:   # event nodes not timeable: time eagerly
        cache.set_timing(True)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for t in range(W + K, W + 2 * K):
                enqueue_step(t)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms_total_b = e0.elapsed_time(e1)
        ktimes = cache.kernel_times()
        timing_mode = "events around eager launches"
    cache.set_timing(False)
    del graph_b
    st2 = cache.stats()
    misses_b = st2["misses"] - st1["misses"]
    hits_b = st2["hits"] - st1["hits"]
    n_launch_per_step = L * (3 if w.shared_kv else 2)   # select + attention (+ merge for latent rows)

    # ---- e2e through the API: host inputs in, host outputs out, every step ------------
    E = args.e2e_steps
    q_pin = torch.from_numpy(q_host.view(np.int16)).pin_memory()
    kv_pin = torch.from_numpy(kv_host.view(np.int16)).pin_memory()
    key_pin = torch.from_numpy(key_host).pin_memory()
    qi_pin = torch.from_numpy(np.ascontiguousarray(walks.transpose(2, 0, 1, 3))).pin_memory()
    out_pin = torch.empty((L, R, w.h_q, w.d_v), dtype=torch.bfloat16).pin_memory()
    qi_d = torch.empty((L, R, w.d_idx), dtype=torch.int8, device=dev)
    q_d = torch.empty((L, R, w.h_q, w.d_qk), dtype=torch.int16, device=dev)
    kv_d = torch.empty((L, R, 1, w.row_elems), dtype=torch.int16, device=dev)
    key_d = torch.empty((L, R, 1, w.d_idx), dtype=torch.int8, device=dev)
    h2d = qi_d.numel() + 2 * q_d.numel() + 2 * kv_d.numel() + key_d.numel()
    d2h = 2 * out_pin.numel()
    e2e_val = None
    if E > 0:
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for t in range(W + 2 * K, W + 2 * K + E):
                qi_d.copy_(qi_pin[t], non_blocking=True)
                q_d.copy_(q_pin[t], non_blocking=True)
                kv_d.copy_(kv_pin[t], non_blocking=True)
                key_d.copy_(key_pin[t], non_blocking=True)
                for l in range(L):
                    cache.decode_layer(l, qi_d[l], q_d[l], out=out_dev[l], stream=stream,
                                       new_kv=kv_d[l], new_keys=key_d[l])
                out_pin.copy_(out_dev, non_blocking=True)
                stream.synchronize()
        e2e_s = max_over_ranks(time.perf_counter() - t0, world)
        e2e_val = world * E * L / e2e_s
    final = cache.stats()
    dev_err = final["device_error"]

    # ---- numbers -------------------------------------------------------------------
    ms_step = ms_total / K
    value = world * K * L / (ms_total * 1e-3)
    tokens = world * K * R / (ms_total * 1e-3)
    # algorithmic traffic of a timed region (contexts grow by one per step)
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def region_bytes(t_begin, n_miss):
        hb = {k: 0.0 for k in KERNEL_FILES}
        lb = {k: 0.0 for k in KERNEL_FILES}
        m_ls = n_miss * max(1, args.page_size) / (K * L)   # rows (page mode: a missed page is P rows)
        rp = resolve_pulls(args.fetch_mode, w.shared_kv)
        for t in range(t_begin, t_begin + K):
            for l in range(L):
                ab = algorithmic_bytes(w, n0 + t + 1, m_ls, rp, selects=l % max(1, args.index_share) == 0,
                                       page_size=args.page_size)
                for k in KERNEL_FILES:
                    hb[k] += ab["hbm"][k]
                    lb[k] += ab["link"][k]
        return hb, lb

    hb_a, lb_a = region_bytes(W, misses)
    hbm_total = sum(hb_a.values())
    link_total = sum(lb_a.values())
    per_kernel_bytes, per_kernel_link = region_bytes(W + K, misses_b)
    peak_hbm, peak_src = measured_peaks()
    peak_link = link_peak_gbs(dev)
    t_roof = max(hbm_total / (peak_hbm * 1e9), link_total / (peak_link * 1e9))
    step_frac = t_roof / (ms_total * 1e-3)
    kernels = {}
    for k, (ms, n) in ktimes.items():
        if n == 0:
            continue
        avg = ms / n
        kernels[k] = {"launches": n, "avg_us": round(avg * 1e3, 3), "share": None,
                      "hbm_gbs": round(per_kernel_bytes[k] / n / (avg * 1e-3) / 1e9, 1),
                      "link_gbs": round(per_kernel_link[k] / n / (avg * 1e-3) / 1e9, 1),
                      "hbm_bytes_per_launch": int(per_kernel_bytes[k] / n),
                      "link_bytes_per_launch": int(per_kernel_link[k] / n)}
    if "attention" in kernels:
        # the attention products on the tensor cores: 2 h_q (d_qk + d_v) flops per
        # selected row (QK^T and PV).  Latent rows sit near the ridge point
        # (~210 flop/byte against ~250 for these peaks); GQA rows far below it.
        k_sum = float(np.minimum(w.top_k, n0 + W + K).sum())
        fl = 2.0 * w.h_q * (w.d_qk + w.d_v) * k_sum
        a = kernels["attention"]
        tf_peak, tf_src = measured_bf16_tflops()
        a["flops_per_launch"] = int(fl)
        a["tflops"] = round(fl / (a["avg_us"] * 1e-6) / 1e12, 1)
        a["tensor_frac"] = round(a["tflops"] / tf_peak, 4)
        a["tensor_peak"] = {"tflops": tf_peak, "source": tf_src}
    tot_k = sum(v["avg_us"] * v["launches"] for v in kernels.values()) or 1.0
    for v in kernels.values():
        v["share"] = round(v["avg_us"] * v["launches"] / tot_k, 4)
    dom = max(kernels, key=lambda k: kernels[k]["share"]) if kernels else None
    roof = None
    if dom:
        kd = kernels[dom]
        if kd["link_bytes_per_launch"] / (peak_link * 1e9) > kd["hbm_bytes_per_launch"] / (peak_hbm * 1e9):
            # the kernel's own bound is the host link (RESOLVE pulling many rows)
            ach = kd["link_gbs"]
            roof = {"kernel": dom, "bound": "link", "achieved": ach, "peak": round(peak_link, 1), "unit": "GB/s",
                    "frac": round(ach / peak_link, 4), "peak_source": "pinned cudaMemcpyAsync H2D, measured in this run",
                    "traffic": ncu_traffic(dom, w.name, w.shared_kv), "traffic_unit": "HBM bytes per launch (ncu)",
                    "bytes_per_launch": kd["link_bytes_per_launch"]}
        else:
            ach = kd["hbm_gbs"]
            roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peak_hbm, "unit": "GB/s",
                    "frac": round(ach / peak_hbm, 4), "peak_source": peak_src,
                    "traffic": ncu_traffic(dom, w.name, w.shared_kv), "bytes_per_launch": kd["hbm_bytes_per_launch"]}
    # latent rows: the attention entry also launches the partial-merge kernel
    gpu_launches = sum(v["launches"] for v in kernels.values()) + (
        kernels.get("attention", {}).get("launches", 0) if w.shared_kv else 0)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "dtype_detail": "int8 indexer (int32 accumulate); bf16 K/V and q, fp32 softmax/accumulate",
        "data": "synthetic (seeded; N(0,1) bf16 K/V, uniform int8 index keys, random-walk int8 queries)",
        "config": workload_config(w, args, world),
        "timed": "one CUDA graph of the timed steps, uploaded beforehand, replayed once"
        if uploaded and uploaded[0] else "one CUDA graph of the timed steps, replayed once (not "
        "uploaded beforehand: this torch does not expose the executable graph)",
        "kernel_timing": {"mode": timing_mode, "steps": K, "ms_per_step": round(ms_total_b / K, 4),
                          "miss_rate": round(misses_b / max(1, hits_b + misses_b), 5),
                          "note": "the K steps after the headline's, each kernel bracketed by CUDA events "
                                  "(the events split the programmatic launches, so kernels do not overlap)"},
        "tokens_per_s": round(tokens, 1),
        "hbm_gbs": round(hbm_total / (ms_total * 1e-3) / 1e9, 1),
        "link_gbs": round(link_total / (ms_total * 1e-3) / 1e9, 2),
        "link_peak_gbs": round(peak_link, 1),
        "miss_rate": round(misses / max(1, hits + misses), 5),
        "full_select_frac": round((st1["full_selects"] - st0["full_selects"]) / max(1, K * L * R), 4),
        "misses_per_layer_step": round(misses / (K * L), 1),
        "attention_timeline": attention_timeline(st0, st1, K * L, torch.cuda.get_device_properties(dev).multi_processor_count),
        "step_roofline": {"t_roof_ms": round(t_roof * 1e3 / K, 4), "t_meas_ms": round(ms_step, 4),
                          "frac": round(step_frac, 4), "hbm_bytes_per_step": int(hbm_total / K),
                          "link_bytes_per_step": int(link_total / K),
                          "bound": "hbm" if hbm_total / peak_hbm >= link_total / peak_link else "link"},
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": gpu_launches if gpu_launches else n_launch_per_step * K,
        "e2e": {"value": round(e2e_val, 2) if e2e_val else None, "unit": UNIT, "steps": E,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "clocks": clk,
        "prefill_s": round(t_pre, 1),
        "host_store": host_pages,
        "device_error": dev_err,
    }
    cache.close()
    if args.policy_floor and args.page_size <= 1 and rank == 0:   # the floor is token-level
        try:   # a report beside the measurement: it must never cost the bench line
            out["policy_floor"] = policy_floor(args, w, dev_index)
        except Exception as e:   # noqa: BLE001
            out["policy_floor"] = {"error": f"{type(e).__name__}: {e}"}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="hisparse", choices=["hisparse", "reference"])
    ap.add_argument("--workload", default="batch16_32k", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--hot-slots", type=int, default=None)
    ap.add_argument("--sigma", type=float, default=None)
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--fetch-mode", type=int, default=2, choices=[0, 1, 2],
                    help="who copies missed rows: 0 the attention kernel (overlapped), 1 RESOLVE, "
                         "2 chosen per request (default)")
    ap.add_argument("--replacement", default="lru", choices=["lru", "fifo", "random"],
                    help="hot-cache replacement: lru (the method's), fifo or random (its comparison policies)")
    ap.add_argument("--index-share", type=int, default=1,
                    help="layers per indexer group: > 1 reuses the group lead's selection in the following "
                         "layers (a variant; the workloads select per layer)")
    ap.add_argument("--share-prefetch", type=int, default=1,
                    help="with --index-share > 1: 1 = the lead's call resolves and pulls the followers ahead, "
                         "0 = each follower resolves at its own call")
    ap.add_argument("--page-size", type=int, default=1,
                    help="Quest-style page selection: pages of this many positions (1 = token-level top-k)")
    ap.add_argument("--policy-floor", type=int, default=1,
                    help="1: also report the policy's misses against Belady's MIN on a cold 2-request trace "
                         "(untimed, after the measurement); 0: skip")
    ap.add_argument("--cpu-sample", default="2x2x100", help="oracle sample: requests x layers x steps")
    ap.add_argument("--clock-interval-ms", type=int, default=10,
                    help="nvidia-smi clock sampling period during the timed region (0: off)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "hisparse" else "gloo"
        dist.init_process_group(backend=backend)

    w = wl.WORKLOADS[args.workload]
    if args.hot_slots or args.sigma is not None:
        w = wl.stress_point(args.hot_slots or w.hot_slots, args.sigma if args.sigma is not None else w.sigma) \
            if args.workload == "stress_128k" else wl.make_workload(
                args.workload, **({"hot_slots": args.hot_slots} if args.hot_slots else {}),
                **({"sigma": args.sigma} if args.sigma is not None else {}))
    w = rank_workload(w, rank, world)

    sr, sl, ss = (int(x) for x in args.cpu_sample.split("x"))
    sr, sl = min(sr, w.n_requests), min(sl, w.n_layers)   # the sample stays inside the workload
    if args.impl == "reference":
        if rank != 0:
            return
        res = run_reference(args, w, sr, sl, ss)
        print(json.dumps(res), flush=True)
        return

    res = run_hisparse(args, w, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            secs, units = oracle_sample(w, range(sr), range(sl), ss, args.replacement)
            per_unit = secs / units
            res["cpu_baseline"] = {"value": round(1.0 / (per_unit * w.n_requests), 4), "unit": UNIT,
                                   "cores": cpu_threads(), "kind": "oracle",
                                   "sample": f"{sr} request(s) x {sl} layer(s) x {ss} decode steps of {w.name} "
                                             f"({units} request-layer-steps, {secs:.1f} s), scaled by "
                                             f"{w.n_requests} requests per layer-step"}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def workload_config(w: wl.Workload, args, world: int) -> dict:
    """The workload and method settings both arms report (the same dict)."""
    n0 = w.contexts()
    ab = algorithmic_bytes(w, n0, 0.0, page_size=args.page_size)   # one layer-step, no misses
    step_mib = w.n_layers * sum(ab["hbm"].values()) / 2**20
    return {"workload": w.name, "requests": w.n_requests, "layers": w.n_layers,
            "context": int(n0[0]) if w.context_range is None else [int(n0.min()), int(n0.max())],
            "h_q": w.h_q, "h_kv": w.h_kv, "d_qk": w.d_qk, "d_v": w.d_v, "d_idx": w.d_idx, "top_k": w.top_k,
            "hot_slots": w.hot_slots, "sigma": w.sigma,
            "parallelism": f"requests sharded, {world} independent cache(s)",
            "l2": f"inputs larger than L2: at least {step_mib:.0f} MiB read per step > 129 MiB",
            "fetch_mode": args.fetch_mode, "replacement": args.replacement,
            **({"index_share": args.index_share, "share_prefetch": args.share_prefetch}
               if args.index_share > 1 else {}),
            **({"page_size": args.page_size} if args.page_size > 1 else {})}


def run_reference(args, w: wl.Workload, sr: int, sl: int, ss: int) -> dict:
    """The CPU oracle as the reference arm: each step runs the oracle on a
    bounded sample (sr requests x sl layers, one decode step each) and the rate
    is scaled to the whole batch."""
    W, K = args.warmup, args.steps
    steps = W + K
    # the oracle replays steps 0..steps-1 of each sampled (request, layer); the
    # first W are the warm-up
    from oracle import indexer_scores_many, sparse_attention, topk_select
    per_step = []
    for l in range(sl):
        for r in range(sr):
            keys = wl.idx_keys_upto(w, r, l, steps)
            walk = wl.query_walk(w, r, l, steps)
            kv = wl.prefill_kv(w, r, l)
            n0 = int(w.contexts()[r])
            cache = oracle_cache(w, r, l, args.replacement)
            for t in range(steps):
                q = wl.step_query(w, r, l, t)
                app = [wl.step_kv_row(w, r, l, u) for u in range(t + 1)]
                t0 = time.perf_counter()
                n = n0 + t + 1
                s = indexer_scores_many(keys[:n], walk[t])[:, 0]
                sel = topk_select(s, w.top_k)
                cache.step(sel)
                rows = np.empty((sel.size, w.row_elems), np.uint16)
                pre = sel < n0
                rows[pre] = kv[sel[pre]]
                for i in np.nonzero(~pre)[0]:
                    rows[i] = app[int(sel[i] - n0)]
                sparse_attention(q, rows, h_kv=w.h_kv, d_qk=w.d_qk, d_v=w.d_v, v_offset=w.v_offset)
                if t >= W:
                    per_step.append(time.perf_counter() - t0)
    per_unit = float(np.mean(per_step))
    value = 1.0 / (per_unit * w.n_requests)
    sample = (f"{sr} request(s) x {sl} layer(s) per step, steps {W}..{steps - 1} of {w.name}, "
              f"scaled by {w.n_requests} requests per layer-step")
    # one step of this arm is the bounded sample (sr x sl request-layer-steps), so
    # ms_per_step is its measured time; value scales the rate to the whole batch
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
            "steps": K, "warmup": W, "ms_per_step": round(per_unit * sr * sl * 1e3, 2),
            "step": f"a sample of {sr} request(s) x {sl} layer(s) of one decode step (value is scaled to "
                    f"{w.n_requests} requests per layer-step)",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": workload_config(w, args, args.gpus),
            "timed": "the CPU oracle (numpy, fp64 / int64) on the host's cores, a bounded sample per step",
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


if __name__ == "__main__":
    main()
