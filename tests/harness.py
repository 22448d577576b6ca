"""Drives the CUDA library through its binding on a synthetic workload and
compares it with the CPU oracle.  Used by the GPU tests and the smoke check."""
from __future__ import annotations

import numpy as np

import workload as wl

# attention tolerance against the fp64 oracle (bf16 output of fp32 accumulation)
MAX_ABS = 2e-2
REL_L2 = 5e-3


def torch_mod():
    import torch
    return torch


def make_cache(w: wl.Workload, steps: int, hot_slots: int | None = None, device: int = 0, fetch_mode: int = 2,
               replacement: str = "lru", replacement_seed: int = 0, write_allocate: bool = False, **extra):
    from tiered_kv_cache_int8_gb300 import HiSparseCache
    return HiSparseCache(n_layers=w.n_layers, max_requests=w.n_requests, max_context=w.max_context(steps),
                         h_q=w.h_q, h_kv=w.h_kv, d_qk=w.d_qk, d_v=w.d_v, d_idx=w.d_idx, top_k=w.top_k,
                         hot_slots=hot_slots or w.hot_slots, shared_kv=w.shared_kv, device=device,
                         fetch_mode=fetch_mode, replacement=replacement, replacement_seed=replacement_seed,
                         write_allocate=write_allocate, idx_heads=w.idx_heads, **extra)


def packed_q_idx(w: wl.Workload, heads: np.ndarray, weights: np.ndarray) -> np.ndarray:
    """The multi-head indexer's query rows as the library takes them: per request
    the heads [H, d_idx], then the H weights, then zero padding to 16 bytes."""
    R, H, d = heads.shape
    out = np.zeros((R, H * d + 16), np.int8)
    out[:, :H * d] = heads.reshape(R, H * d)
    out[:, H * d:H * d + H] = weights
    return out


def prefill(cache, w: wl.Workload, requests=None, layers=None):
    """Appends every request's initial context through hs_append (one call per
    (request, layer), rows staged in device memory)."""
    torch = torch_mod()
    dev = torch.device("cuda", cache.device)
    requests = range(w.n_requests) if requests is None else requests
    layers = range(w.n_layers) if layers is None else layers
    for l in layers:
        for r in requests:
            kv = wl.prefill_kv(w, r, l)
            keys = wl.prefill_idx_keys(w, r, l)
            kv_t = torch.from_numpy(kv.view(np.int16)).to(dev).view(1, kv.shape[0], kv.shape[1])
            k_t = torch.from_numpy(keys).to(dev).view(1, keys.shape[0], keys.shape[1])
            rid = torch.tensor([r], dtype=torch.int32, device=dev)
            cache.append(l, kv_t, k_t, req_ids=rid)
    torch.cuda.synchronize(dev)


class StepInputs:
    """Per-step inputs of all requests of one layer, on the device."""

    def __init__(self, w: wl.Workload, steps: int, device: int = 0, layers=None):
        torch = torch_mod()
        dev = torch.device("cuda", device)
        self.w = w
        layers = range(w.n_layers) if layers is None else layers
        R = w.n_requests
        self.walk = {l: np.stack([wl.query_walk(w, r, l, steps) for r in range(R)]) for l in layers}
        if w.idx_heads > 1:   # every head's walk [R, T, H, d] and the per-step weights [R, T, H]
            self.heads = {l: np.stack([wl.query_walk_heads(w, r, l, steps) for r in range(R)]) for l in layers}
            self.weights = {l: np.stack([np.stack([wl.step_idx_weights(w, r, l, t) for t in range(steps)])
                                         for r in range(R)]) for l in layers}
        self.q_idx = {}
        self.q = {}
        self.kv = {}
        self.keys = {}
        for l in layers:
            for t in range(steps):
                if w.idx_heads > 1:
                    qi = packed_q_idx(w, self.heads[l][:, t], self.weights[l][:, t])
                else:
                    qi = np.ascontiguousarray(self.walk[l][:, t])
                self.q_idx[l, t] = torch.from_numpy(qi).to(dev)
                q = np.stack([wl.step_query(w, r, l, t) for r in range(R)])
                self.q[l, t] = torch.from_numpy(q.view(np.int16)).to(dev)
                kv = np.stack([wl.step_kv_row(w, r, l, t) for r in range(R)])[:, None, :]
                self.kv[l, t] = torch.from_numpy(np.ascontiguousarray(kv).view(np.int16)).to(dev)
                k = np.stack([wl.step_idx_key(w, r, l, t) for r in range(R)])[:, None, :]
                self.keys[l, t] = torch.from_numpy(np.ascontiguousarray(k)).to(dev)


def run_steps(cache, w: wl.Workload, inp: StepInputs, steps: int, layers=None, *, collect_sel=True,
              collect_out=True, collect_meta=False, t0: int = 0, fused: bool = False, meta_pairs=None):
    """Runs decode steps t0..t0+steps-1 (append then decode per layer; with
    fused=True the append rides on the decode call); returns per-(layer, step)
    selections, outputs and (optionally) metadata snapshots: of every request,
    or with meta_pairs = {(request, layer), ...} of those only (a dict per step)."""
    torch = torch_mod()
    dev = torch.device("cuda", cache.device)
    layers = range(w.n_layers) if layers is None else layers
    R = w.n_requests
    res = {"sel": {}, "out": {}, "meta": {}}
    for t in range(t0, t0 + steps):
        for l in layers:
            sel = torch.full((R, w.top_k), -7, dtype=torch.int32, device=dev)
            if fused:
                out = cache.decode_layer(l, inp.q_idx[l, t], inp.q[l, t], sel_out=sel, new_kv=inp.kv[l, t],
                                         new_keys=inp.keys[l, t])
            else:
                cache.append(l, inp.kv[l, t], inp.keys[l, t])
                out = cache.decode_layer(l, inp.q_idx[l, t], inp.q[l, t], sel_out=sel)
            if collect_sel:
                res["sel"][l, t] = sel.cpu().numpy()
            if collect_out:
                res["out"][l, t] = out.view(torch.int16).cpu().numpy().view(np.uint16)
            if collect_meta:
                n0 = w.contexts()
                res["meta"][l, t] = [cache.snapshot(r, l, int(n0[r]) + t + 1) for r in range(R)]
            elif meta_pairs:
                n0 = w.contexts()
                res["meta"][l, t] = {r: cache.snapshot(r, l, int(n0[r]) + t + 1)
                                     for (r, ll) in meta_pairs if ll == l}
    torch.cuda.synchronize(dev)
    return res


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def attention_error(gpu_bits: np.ndarray, ref: np.ndarray):
    g = bf16_bits_to_f64(gpu_bits)
    max_abs = float(np.abs(g - ref).max())
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    return max_abs, rel
