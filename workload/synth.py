"""Seeded synthetic workloads.

The HiSparse pages (HiSparse deep summary, "KV卸载上主机" column; HiSparse study
notes, "方法") measure on real models and serving traces that are not available
here.  These generators stand in for them with the shapes and distributions of
the five benchmark workloads:

* prefill K/V rows ~ N(0, 1), stored as bf16 (round-to-nearest-even of a float32
  sample, done on the bit pattern);
* index keys uniform int8 in [-127, 127];
* one int8 indexer query per (request, layer, step), a random walk on the unit
  sphere quantised to [-127, 127], so consecutive steps select overlapping
  positions (the locality the pages rely on for LRU);
* attention queries ~ N(0, 1) bf16, independent of the indexer query;
* one appended token per (request, layer, step) drawn from the same
  distributions as the prefill.

Every array comes from its own counter-addressed numpy stream
``SeedSequence(seed, spawn_key=(request, layer, stream, index))``, so any
piece can be regenerated on its own (the oracle checks sampled requests at full
size without holding the whole store) and the result does not depend on the
number of threads.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np

# stream ids inside a (request, layer) key
_S_PREFILL_KV = 0
_S_PREFILL_IDX = 1
_S_WALK = 2
_S_QUERY = 3
_S_STEP_KV = 4
_S_STEP_IDX = 5
_S_LENGTHS = 6
_S_IDX_W = 7             # per-step indexer head weights (multi-head indexer)

KV_CHUNK = 4096          # positions per prefill K/V stream
IDX_CHUNK = 65536        # positions per prefill index-key stream


@dataclass(frozen=True)
class Workload:
    name: str
    seed_index: int              # distinct per workload: the default seed is 20260000 + seed_index
    n_requests: int
    n_layers: int
    context: int                 # initial context per request (fixed-length workloads)
    h_q: int
    h_kv: int
    d_qk: int
    d_v: int
    shared_kv: bool              # latent row read as K (all d_qk) and V (first d_v)
    d_idx: int
    top_k: int
    hot_slots: int
    steps: int
    sigma: float
    context_range: tuple | None = None   # (lo, hi): per-request log-uniform lengths
    noise: str = "per_dim"       # "per_dim": eps ~ N(0, I/d_idx); "literal": eps ~ N(0, I)
    seed: int | None = None
    idx_heads: int = 1           # > 1: the multi-head ReLU-weighted indexer (one walk per head)

    # ---- derived layout -------------------------------------------------
    @property
    def row_elems(self) -> int:
        """bf16 elements in one position's K/V row (all kv heads of one layer)."""
        if self.shared_kv:
            return self.d_qk
        return self.h_kv * (self.d_qk + self.d_v)

    @property
    def row_bytes(self) -> int:
        return 2 * self.row_elems

    @property
    def v_offset(self) -> int:
        """Element offset of the V region inside a row."""
        return 0 if self.shared_kv else self.h_kv * self.d_qk

    @property
    def base_seed(self) -> int:
        return self.seed if self.seed is not None else 20260000 + self.seed_index

    def contexts(self) -> np.ndarray:
        """Initial context length of every request (int64 [R])."""
        if self.context_range is None:
            return np.full(self.n_requests, self.context, dtype=np.int64)
        lo, hi = self.context_range
        g = _rng(self.base_seed, (0, 0, _S_LENGTHS, 0))
        u = g.uniform(math.log(lo), math.log(hi), size=self.n_requests)
        return np.rint(np.exp(u)).astype(np.int64)

    def max_context(self, extra_steps: int | None = None) -> int:
        t = self.steps if extra_steps is None else extra_steps
        return int(self.contexts().max()) + t

    def host_bytes(self) -> int:
        """Bytes of the authoritative host copy at the end of the run."""
        return int((self.contexts() + self.steps).sum()) * self.n_layers * self.row_bytes

    def hot_bytes(self) -> int:
        return self.n_requests * self.n_layers * self.hot_slots * self.row_bytes


def _rng(seed: int, key: tuple) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=key)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest, ties to even.

    Inputs are finite samples; NaN handling is not needed for generation."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(g: np.random.Generator, shape) -> np.ndarray:
    x = g.standard_normal(size=shape, dtype=np.float32)
    return f32_to_bf16_bits(x)


def _uniform_i8(g: np.random.Generator, shape) -> np.ndarray:
    return g.integers(-127, 128, size=shape, dtype=np.int8)


_POOL: ThreadPoolExecutor | None = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1))
    return _POOL


# ---- prefill ----------------------------------------------------------------

def prefill_kv(w: Workload, req: int, layer: int, out: np.ndarray | None = None,
               parallel: bool = True) -> np.ndarray:
    """K/V rows of positions [0, N0_r) of one (request, layer): uint16 [N0_r, row_elems]."""
    n = int(w.contexts()[req])
    if out is None:
        out = np.empty((n, w.row_elems), dtype=np.uint16)
    assert out.shape == (n, w.row_elems) and out.dtype == np.uint16
    seed = w.base_seed

    def fill(c):
        lo = c * KV_CHUNK
        hi = min(n, lo + KV_CHUNK)
        g = _rng(seed, (req, layer, _S_PREFILL_KV, c))
        out[lo:hi] = _normal_bf16(g, (hi - lo, w.row_elems))

    chunks = range((n + KV_CHUNK - 1) // KV_CHUNK)
    if parallel and len(chunks) > 1:
        list(_pool().map(fill, chunks))
    else:
        for c in chunks:
            fill(c)
    return out


def prefill_idx_keys(w: Workload, req: int, layer: int) -> np.ndarray:
    """Index keys of positions [0, N0_r): int8 [N0_r, d_idx]."""
    n = int(w.contexts()[req])
    out = np.empty((n, w.d_idx), dtype=np.int8)
    for c in range((n + IDX_CHUNK - 1) // IDX_CHUNK):
        lo = c * IDX_CHUNK
        hi = min(n, lo + IDX_CHUNK)
        out[lo:hi] = _uniform_i8(_rng(w.base_seed, (req, layer, _S_PREFILL_IDX, c)), (hi - lo, w.d_idx))
    return out


# ---- per-step inputs ----------------------------------------------------------

def query_walk_heads(w: Workload, req: int, layer: int, steps: int | None = None) -> np.ndarray:
    """Indexer queries of every head for steps 0..T-1: int8 [T, idx_heads, d_idx].
    Head 0 is query_walk's walk; head h > 0 is an independent walk of its own
    stream, with the same sigma."""
    T = w.steps if steps is None else steps
    heads = [query_walk(w, req, layer, T)]
    for h in range(1, w.idx_heads):
        heads.append(_walk(w, _rng(w.base_seed, (req, layer, _S_WALK, h)), T))
    return np.stack(heads, axis=1)


def step_idx_weights(w: Workload, req: int, layer: int, t: int) -> np.ndarray:
    """Per-head indexer weights of one (request, layer, step): int8 [idx_heads]
    uniform in [0, 127] (the multi-head indexer's query-dependent weights)."""
    return _rng(w.base_seed, (req, layer, _S_IDX_W, t)).integers(0, 128, size=w.idx_heads, dtype=np.int8)


def _walk(w: Workload, g: np.random.Generator, T: int) -> np.ndarray:
    d = w.d_idx
    u = g.standard_normal(d)
    u /= np.linalg.norm(u)
    eps_scale = 1.0 / math.sqrt(d) if w.noise == "per_dim" else 1.0
    out = np.empty((T, d), dtype=np.int8)
    for t in range(T):
        if t > 0:
            u = u + w.sigma * eps_scale * g.standard_normal(d)
            u /= np.linalg.norm(u)
        q = np.rint(127.0 * u / np.abs(u).max())
        out[t] = np.clip(q, -127, 127).astype(np.int8)
    return out


def query_walk(w: Workload, req: int, layer: int, steps: int | None = None) -> np.ndarray:
    """Indexer queries for decode steps 0..T-1 of one (request, layer): int8 [T, d_idx].

    u_0 = normalise(N(0, I)); u_t = normalise(u_{t-1} + sigma * eps_t);
    q_t = round_half_even(127 * u_t / max|u_t|).  eps_t ~ N(0, I / d_idx) under
    the per-dimension reading (drift of about sigma radians per step), N(0, I)
    under the literal one."""
    T = w.steps if steps is None else steps
    return _walk(w, _rng(w.base_seed, (req, layer, _S_WALK, 0)), T)


def step_query(w: Workload, req: int, layer: int, t: int) -> np.ndarray:
    """Attention query of one (request, layer, step): bf16 bits uint16 [H_q, d_qk]."""
    return _normal_bf16(_rng(w.base_seed, (req, layer, _S_QUERY, t)), (w.h_q, w.d_qk))


def step_kv_row(w: Workload, req: int, layer: int, t: int) -> np.ndarray:
    """K/V row of the token appended before decode step t: uint16 [row_elems]."""
    return _normal_bf16(_rng(w.base_seed, (req, layer, _S_STEP_KV, t)), (w.row_elems,))


def step_idx_key(w: Workload, req: int, layer: int, t: int) -> np.ndarray:
    """Index key of the token appended before decode step t: int8 [d_idx]."""
    return _uniform_i8(_rng(w.base_seed, (req, layer, _S_STEP_IDX, t)), (w.d_idx,))


def kv_rows_at(w: Workload, req: int, layer: int, positions: np.ndarray) -> np.ndarray:
    """K/V rows of arbitrary positions (prefill or appended) of one (request, layer)."""
    positions = np.asarray(positions, dtype=np.int64)
    n0 = int(w.contexts()[req])
    out = np.empty((positions.size, w.row_elems), dtype=np.uint16)
    pre = positions < n0
    if pre.any():
        for c in np.unique(positions[pre] // KV_CHUNK):
            lo = int(c) * KV_CHUNK
            hi = min(n0, lo + KV_CHUNK)
            block = _normal_bf16(_rng(w.base_seed, (req, layer, _S_PREFILL_KV, int(c))), (hi - lo, w.row_elems))
            m = pre & (positions // KV_CHUNK == c)
            out[m] = block[positions[m] - lo]
    for i in np.nonzero(~pre)[0]:
        out[i] = step_kv_row(w, req, layer, int(positions[i] - n0))
    return out


def idx_keys_upto(w: Workload, req: int, layer: int, n_steps: int) -> np.ndarray:
    """All index keys after n_steps appends: int8 [N0_r + n_steps, d_idx]."""
    pre = prefill_idx_keys(w, req, layer)
    if n_steps == 0:
        return pre
    app = np.stack([step_idx_key(w, req, layer, t) for t in range(n_steps)])
    return np.concatenate([pre, app])


# ---- the benchmark workloads ---------------------------------------------------

WORKLOADS: dict[str, Workload] = {
    # 1 request x 1 layer, context 4096, d_idx 64, k 256, B 512, 32 steps
    "tiny": Workload("tiny", 1, 1, 1, 4096, 8, 1, 128, 128, False, 64, 256, 512, 32, 0.1),
    # batch 16, 4 layers, 32K context, GQA 32/8/128, k 2048, B 4096, 64 steps
    "batch16_32k": Workload("batch16_32k", 2, 16, 4, 32768, 32, 8, 128, 128, False, 128, 2048, 4096, 64, 0.1),
    # batch 32, 2 layers, 128K, one 576-wide latent row (first 512 = V), 128 heads
    "mla_128k": Workload("mla_128k", 3, 32, 2, 131072, 128, 1, 576, 512, True, 128, 2048, 4096, 32, 0.1),
    # 64 requests, context log-uniform in [8K, 200K], 2 layers, GQA
    "mixed_8k_200k": Workload("mixed_8k_200k", 4, 64, 2, 0, 32, 8, 128, 128, False, 128, 2048, 4096, 32, 0.1,
                              context_range=(8192, 204800)),
    # batch 64 at 128K, 2 layers, GQA; swept over B and sigma
    "stress_128k": Workload("stress_128k", 5, 64, 2, 131072, 32, 8, 128, 128, False, 128, 2048, 4096, 64, 0.1),
}

STRESS_B = (2048, 4096, 8192)
STRESS_SIGMA = (0.05, 0.1, 0.3)


def stress_point(B: int, sigma: float) -> Workload:
    return replace(WORKLOADS["stress_128k"], hot_slots=B, sigma=sigma,
                   name=f"stress_128k_B{B}_s{sigma}")


def make_workload(base: str, **over) -> Workload:
    """A workload with some fields replaced (smaller parity cases keep the
    base's distributions and seed)."""
    w = WORKLOADS[base]
    if "name" not in over:
        over["name"] = base + "_" + "_".join(f"{k}{v}" for k, v in sorted(over.items()))
    return replace(w, **over)
