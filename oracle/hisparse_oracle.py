"""Plain CPU oracle for one decode layer-step of top-k sparse attention over a
two-level KV cache (HiSparse).

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import or run this module.  The CUDA library never calls
it and shares no code with it; the two meet only at the seeded input generators
in the ``workload`` package.

What is computed, and where it is stated:

* "KV卸载上主机:HiSparse、PDD与DDR4回收" (yeyulingfeng.com), section
  "二、论文分析 / 论文1：HiSparse": an indexer tells every step which KV
  positions it needs; the authoritative full KV lives in pinned host DRAM, the GPU
  keeps B slots per request per layer, a page table plus LRU metadata drive
  replacement, and only placement changes, so the result is exactly top-k sparse
  attention over the full KV.
* "10月14日学习笔记" (zgchen.com), section "HiSparse / 动机": the indexer picks
  the top-k tokens; "方法" item 1: adjacent decode steps overlap, LRU fits best.
* "Heterogeneous LLM Serving with General-Purpose Processing-Near-Memory for
  Retrieval-Based Sparse Attention" (vsvnakers.github.io), section
  "核心公式与算法", formula 2: Attention = softmax(QK^T / sqrt(d_k) (masked)) V.
  The mask is printed as an elementwise product; read here as an additive
  -inf mask, i.e. softmax over the selected positions only.

Steps the pages leave open are fixed as follows (each is one plain reading):
indexer = one int8 query dot int8 index key, exact integer sum, no scale;
candidates = every position < N including the token just appended;
k_eff = min(k, N); ties broken by lower position; selection reported in
ascending position order; LRU victims = unpinned slots with the smallest
(last-use stamp, slot); misses filled in ascending position order; appends do
not enter the hot cache (write-around), or, under the write-allocate variant,
the token a decode call appends counts as used by that call; q head h reads kv
head floor(h * H_kv / H_q);
softmax scale 1/sqrt(d_qk) unless given.

Floating point is fp64 throughout; integer work is exact int64.
"""
from __future__ import annotations

import heapq
import math

import numpy as np

# ---------------------------------------------------------------------------
# bf16 inputs
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# a1: indexer scores (HiSparse summary: the sparse selector states which
# positions each step needs; the score is fixed here as int8 . int8 -> integer)
# ---------------------------------------------------------------------------


def indexer_scores(idx_keys: np.ndarray, q_idx: np.ndarray) -> np.ndarray:
    """s[p] = sum_j q_idx[j] * K_idx[p, j] for every stored position p, exact int64."""
    k = np.asarray(idx_keys, dtype=np.int8).astype(np.int64)
    q = np.asarray(q_idx, dtype=np.int8).astype(np.int64)
    return k @ q


def indexer_scores_many(idx_keys: np.ndarray, q_idx: np.ndarray) -> np.ndarray:
    """Scores of every position for several queries at once: int64 [N, T].

    Uses a float32 matrix product.  Each product term is at most 128*128 = 2^14
    in magnitude and d_idx <= 1023 terms are summed, so every partial sum is an
    integer below 2^24 and is represented exactly in float32 whatever order the
    library sums in; the result is the exact integer score."""
    k = np.asarray(idx_keys, dtype=np.int8)
    q = np.asarray(q_idx, dtype=np.int8)
    if q.ndim == 1:
        q = q[:, None]
    elif q.shape[0] != k.shape[1]:
        q = q.T
    assert k.shape[1] * 128 * 128 < (1 << 24), "float32 path is exact only for d_idx < 1024"
    s = k.astype(np.float32) @ q.astype(np.float32)
    return s.astype(np.int64)


def indexer_scores_multihead(idx_keys: np.ndarray, q_heads: np.ndarray, weights: np.ndarray) -> np.ndarray:
    """The multi-head ReLU-weighted indexer variant: s[p] = sum_h w_h *
    max(0, q_h . K_idx[p]), exact int64.

    "10月14日学习笔记", "HiSparse / 动机" names the indexer only and the pages
    cite DeepSeek's sparse attention (DSA) without its formula; this reading
    takes DSA's indexer shape: several query heads against one shared key per
    position, each head's dot product through a ReLU, combined with per-head
    non-negative weights.  q_heads: int8 [H, d_idx]; weights: int8 [H] in [0, 127]."""
    k = np.asarray(idx_keys, dtype=np.int8).astype(np.int64)
    q = np.asarray(q_heads, dtype=np.int8).astype(np.int64)
    wts = np.asarray(weights, dtype=np.int8).astype(np.int64)
    assert (wts >= 0).all(), "head weights are non-negative"
    dots = k @ q.T                                   # [N, H]
    return np.maximum(dots, 0) @ wts


# ---------------------------------------------------------------------------
# a2: top-k selection ("10月14日学习笔记", HiSparse / 动机: the indexer keeps
# the top-k tokens).  Ties go to the lower position; output ascending.
# ---------------------------------------------------------------------------


def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Positions of the k_eff = min(k, N) highest scores, ascending (int64)."""
    s = np.asarray(scores, dtype=np.int64)
    n = s.shape[0]
    k_eff = min(k, n)
    pos = np.arange(n, dtype=np.int64)
    order = np.lexsort((pos, -s))          # primary: score desc; secondary: position asc
    return np.sort(order[:k_eff])


# ---------------------------------------------------------------------------
# Quest-style page-granular selection (the HiSparse summary reports its results for
# Qwen3 with Quest page selection as well as for token-level top-k).  Quest is
# named there without its formulas; the reading here: positions are grouped into
# pages of P; a page keeps the element-wise minimum and maximum of its index
# keys; its score is the upper bound of q . k over the page that those give; the
# k // P best pages are selected (ties to the lower page) and every position of
# them is attended.
# ---------------------------------------------------------------------------


def page_bounds(idx_keys: np.ndarray, page_size: int):
    """Element-wise (min, max) of each page's index keys: two int8 [n_pages, d_idx]."""
    k = np.asarray(idx_keys, dtype=np.int8)
    n = k.shape[0]
    n_pages = (n + page_size - 1) // page_size
    kmin = np.empty((n_pages, k.shape[1]), np.int8)
    kmax = np.empty((n_pages, k.shape[1]), np.int8)
    for j in range(n_pages):
        blk = k[j * page_size:min(n, (j + 1) * page_size)]
        kmin[j] = blk.min(axis=0)
        kmax[j] = blk.max(axis=0)
    return kmin, kmax


def page_scores(kmin: np.ndarray, kmax: np.ndarray, q_idx: np.ndarray) -> np.ndarray:
    """U[j] = sum_d max(q_d * kmin[j, d], q_d * kmax[j, d]): the largest q . k any
    key within the page's per-dimension bounds can reach (exact int64)."""
    q = np.asarray(q_idx, dtype=np.int8).astype(np.int64)
    lo = np.asarray(kmin, dtype=np.int8).astype(np.int64) * q
    hi = np.asarray(kmax, dtype=np.int8).astype(np.int64) * q
    return np.maximum(lo, hi).sum(axis=1)


def page_select(idx_keys: np.ndarray, q_idx: np.ndarray, page_size: int, k: int):
    """(pages, positions): the k // page_size pages with the largest bound (ties to
    the lower page), ascending, and all their positions below N, ascending."""
    kmin, kmax = page_bounds(idx_keys, page_size)
    pages = topk_select(page_scores(kmin, kmax, q_idx), k // page_size)
    n = np.asarray(idx_keys).shape[0]
    pos = [p for j in pages for p in range(int(j) * page_size, min(n, (int(j) + 1) * page_size))]
    return pages, np.asarray(pos, dtype=np.int64)


# ---------------------------------------------------------------------------
# a3/a4: the hot cache with LRU replacement (HiSparse summary: fixed B slots per
# request per layer, page table + LRU metadata; study notes "方法" item 1: LRU).
# ---------------------------------------------------------------------------


class LRUHotCache:
    """B-slot hot cache of one (request, layer), kept as plain Python lists.

    State, as the pages name it: a page table position -> slot, the reverse map
    slot -> position, and a last-use stamp per slot (the step counter of the
    decode call that last used it; -1 for a slot never filled).  The step
    counter starts at 0 and grows by one per decode call.

    One decode call with selection ``sel`` (ascending positions):
      1. a selected position with a page-table entry is a hit; its slot is pinned;
      2. the other selected positions are misses, taken in ascending position order;
      3. the victims are the m unpinned slots with the smallest (stamp, slot),
         taken in that order; miss j goes to victim j;
      4. a victim's old position (if any) leaves the page table; the page table and
         reverse map record the new position;
      5. every slot used by the call (hits and fills) gets stamp = step; step += 1.
    Empty slots carry stamp -1, so they fill first, lowest slot first.
    """

    refresh_hits = True   # LRU: a hit renews its slot's stamp

    def __init__(self, n_slots: int):
        self.B = int(n_slots)
        self.slot_pos = [-1] * self.B
        self.slot_stamp = [-1] * self.B
        self.page: dict[int, int] = {}
        self.step_no = 0

    def step(self, sel, allocate: int | None = None) -> dict:
        """One decode call.  ``allocate``: under write-allocate, the position this
        call appended (the highest so far); the cache then treats it as used at
        this step even when the selection does not take it — the update runs over
        sel + [allocate], so an unselected new token is filled into the last
        victim and stamped like the rest.  Hits and misses count the selected
        positions only; such a fill is counted in "allocs" (its row comes with
        the append, not over the host link)."""
        sel = [int(p) for p in sel]
        assert all(a < b for a, b in zip(sel, sel[1:])), "selection must be ascending and unique"
        used = sel
        if allocate is not None and int(allocate) not in sel:
            assert not sel or int(allocate) > sel[-1], "the appended position is the highest"
            used = sel + [int(allocate)]
        assert len(used) <= self.B, "every selected row (and an allocated one) must fit in the hot cache"
        t = self.step_no
        hit_slots = {self.page[p] for p in used if p in self.page}
        misses = [p for p in used if p not in self.page]
        victims = self._victims(t, hit_slots, len(misses))
        fills = []
        for p, v in zip(misses, victims):
            old = self.slot_pos[v]
            if old >= 0:
                del self.page[old]
            self.slot_pos[v] = p
            self.page[p] = v
            fills.append((p, v))
        slot_of_sel = [self.page[p] for p in sel]
        filled = {v for _, v in fills}
        for s in [self.page[p] for p in used]:
            if self.refresh_hits or s in filled:
                self.slot_stamp[s] = t
        self.step_no = t + 1
        allocs = len(used) - len(sel)
        return {
            "slot_of_sel": np.asarray(slot_of_sel, dtype=np.int64),
            "hits": len(sel) - (len(misses) - allocs),
            "misses": len(misses) - allocs,
            "allocs": allocs,
            "fills": fills,
        }

    def _victims(self, t: int, hit_slots: set, m: int) -> list:
        """The m unpinned slots with the smallest (stamp, slot), in that order."""
        candidates = sorted((self.slot_stamp[s], s) for s in range(self.B) if s not in hit_slots)
        return [s for _, s in candidates[:m]]

    def snapshot(self, n_positions: int):
        """(page[n_positions], reverse[B], stamp[B], step) as int64 arrays / int."""
        page = np.full(n_positions, -1, dtype=np.int64)
        for p, s in self.page.items():
            if p < n_positions:
                page[p] = s
        return (page, np.asarray(self.slot_pos, dtype=np.int64),
                np.asarray(self.slot_stamp, dtype=np.int64), self.step_no)


class FIFOHotCache(LRUHotCache):
    """The same hot cache under first-in-first-out replacement, the comparison
    policy of the HiSparse summary's miss-rate ablation ("论文1：HiSparse": LRU
    13.4 % against FIFO 17.2 % at B = 4096).

    Identical to the LRU rule except step 5: only the slots filled by the call
    take stamp = step; a hit keeps the stamp of its fill, so the victims are the
    unpinned slots filled longest ago (smallest (fill stamp, slot)).
    """

    refresh_hits = False


MASK64 = (1 << 64) - 1


def splitmix64(state: int, draw: int) -> int:
    """Output number ``draw`` (1, 2, ...) of SplitMix64 started from ``state``
    (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
    OOPSLA 2014; increment and finaliser constants of Vigna's reference code):
    z = state + draw * 0x9E3779B97F4A7C15, then two xor-shift-multiply rounds and a
    final xor-shift, all modulo 2^64."""
    z = (state + draw * 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


class RandomHotCache(LRUHotCache):
    """The same hot cache under random replacement, the other comparison policy of
    the HiSparse summary's ablation ("论文1：HiSparse": random 16.1 % misses at
    B = 4096).  The pages give no generator; this one is counter-based so that any
    implementation reproduces it: at decode call t of (request, layer), slot s gets
    key = the top 23 bits of splitmix64(seed, counter + 1) with counter =
    ((request * n_layers + layer) << 40) | ((t mod 2^24) << 16) | s.  Never-filled
    slots go first (lowest slot first), as under LRU and FIFO; the rest of the m
    victims are the unpinned filled slots with the smallest (key, slot) — a
    uniformly random subset of them.  Miss j (ascending position) goes to the j-th
    victim in ascending slot order.  Stamps as for LRU (they do not steer this
    policy)."""

    def __init__(self, n_slots: int, *, seed: int, request: int, layer: int, n_layers: int):
        super().__init__(n_slots)
        self.seed = int(seed) & MASK64
        self.rl = int(request) * int(n_layers) + int(layer)

    def key(self, t: int, slot: int) -> int:
        counter = (self.rl << 40) | ((t & 0xFFFFFF) << 16) | slot
        return splitmix64(self.seed, counter + 1) >> 41

    def _victims(self, t: int, hit_slots: set, m: int) -> list:
        ranked = sorted(((0, 0, s) if self.slot_pos[s] < 0 else (1, self.key(t, s), s))
                        for s in range(self.B) if s not in hit_slots)
        return sorted(s for *_, s in ranked[:m])


# ---------------------------------------------------------------------------
# Belady's MIN (HiSparse summary quotes the offline optimum as the floor of the
# LRU miss rate).  A per-step set trace is serialised step by step, ascending
# inside a step; any batched schedule is also a serial one, so MIN of the
# serial trace is a lower bound on every replacement policy's misses.
# ---------------------------------------------------------------------------


def belady_misses(trace, n_slots: int) -> int:
    """Misses of the offline optimum (evict the resident position whose next use
    is farthest; never-used-again counts as infinitely far) on the serialised trace."""
    assert n_slots >= 1
    seq = [int(p) for step in trace for p in sorted(step)]
    n = len(seq)
    nxt = [n] * n
    last: dict[int, int] = {}
    for i in range(n - 1, -1, -1):
        nxt[i] = last.get(seq[i], n + 1 + i)   # distinct "never" values keep the heap total
        last[seq[i]] = i
    resident: dict[int, int] = {}              # position -> its next use
    heap: list = []                            # (-next_use, position), lazily invalidated
    misses = 0
    for i, p in enumerate(seq):
        if p not in resident:
            misses += 1
            if len(resident) >= n_slots:
                while True:
                    negnu, q = heapq.heappop(heap)
                    if resident.get(q) == -negnu:
                        del resident[q]
                        break
        resident[p] = nxt[i]
        heapq.heappush(heap, (-nxt[i], p))
    return misses


# ---------------------------------------------------------------------------
# a5: sparse attention over the selected rows (KARAT digest, formula 2, with
# the mask read as "selected positions only"; HiSparse summary: exact).
# ---------------------------------------------------------------------------


def sparse_attention(q_bits: np.ndarray, rows_bits: np.ndarray, *, h_kv: int, d_qk: int,
                     d_v: int, v_offset: int, scale: float | None = None) -> np.ndarray:
    """o[h] = sum_i softmax_i(scale * q[h] . K_i) V_i over the given rows, fp64.

    q_bits: bf16 bits [H_q, d_qk]; rows_bits: bf16 bits [n, row_elems] in the order
    selected.  K of kv head g = row[g*d_qk : (g+1)*d_qk]; V of kv head g =
    row[v_offset + g*d_v : v_offset + (g+1)*d_v].  q head h reads kv head
    floor(h * h_kv / H_q).  Returns float64 [H_q, d_v]; zeros when n == 0."""
    q = bf16_to_f64(q_bits)
    rows = bf16_to_f64(rows_bits)
    h_q = q.shape[0]
    if scale is None or scale == 0.0:
        scale = 1.0 / math.sqrt(d_qk)
    out = np.zeros((h_q, d_v), dtype=np.float64)
    if rows.shape[0] == 0:
        return out
    for h in range(h_q):
        g = (h * h_kv) // h_q
        K = rows[:, g * d_qk:(g + 1) * d_qk]
        V = rows[:, v_offset + g * d_v: v_offset + (g + 1) * d_v]
        logits = scale * (K @ q[h])
        w = np.exp(logits - logits.max())
        out[h] = (w / w.sum()) @ V
    return out


# ---------------------------------------------------------------------------
# capacity (HiSparse summary: 128K GLM-5.1 request, 13.09 GB BF16 KV, ~0.4 GB
# at B = 4096, about 30x)
# ---------------------------------------------------------------------------


def hot_over_full(n_slots: int, n_positions: int) -> float:
    """Fraction of a request-layer's KV bytes that the hot cache holds: B / N."""
    return n_slots / n_positions


def hot_cache_bytes(full_kv_bytes: float, n_positions: int, n_slots: int) -> float:
    return full_kv_bytes * hot_over_full(n_slots, n_positions)
