// Top-k selection and RESOLVE, one CTA per request.
//
// Method.  "10月14日学习笔记" (zgchen.com), "HiSparse / 动机": attention runs
// over the top-k positions the indexer picks (ties here: the lower position;
// output ascending).  "KV卸载上主机:HiSparse、PDD与DDR4回收", "论文1：HiSparse":
// a page table plus LRU metadata drive replacement of the B hot slots of each
// (request, layer); hit detection, LRU replacement, metadata update and the host
// fetch are resolved in one kernel per layer.  "10月14日学习笔记", "方法" 1: LRU.
//
// Replacement rule: slots holding a selected position (hits) are pinned; the m
// misses, in ascending position order, go to the m unpinned slots with the
// smallest (stamp, slot), in that order; every used slot's stamp (LRU), or only
// every filled slot's (FIFO, a comparison policy of the pages), becomes the
// (request, layer) step counter, which then grows by one.  Random replacement (the
// other comparison policy) takes the m unpinned slots with the smallest
// counter-based hash keys instead, in ascending slot order, and stamps as LRU.
//
// Design (sm_103a), one 1024-thread CTA per request; a latency-bound chain, so
// every global read the chain needs is issued up front, and the steps between
// are shared-memory work:
//  0. prefetch (cp.async): the first-digit histogram the score kernel built, the
//     LRU list, the reverse map (when it fits) and the appended token's row.
//  1. exact top-k over the 24-bit keys the score kernel left in L2, in ONE
//     coalesced pass: the first digit b1 comes from the histogram; each warp
//     scans a contiguous range of positions, four keys per lane per load, and
//     turns "digit above b1" into a bitmap (each 8-lane group's 4-bit nibbles
//     OR-reduced into one 32-position word), while the few keys with digit b1 go
//     to a per-warp list in position order (warp prefix sums) and into the
//     second-digit histogram.  The threshold key and the number of equal keys to
//     take follow from the second histogram; a scan of per-warp counts gives
//     each warp its output offset, and each lane emits the positions of one
//     bitmap word, taking keys equal to the threshold in position order.
//     Contexts above FAST_MAX_N, or a warp whose list overflows (heavy ties),
//     take the same steps with a second and third read of the keys instead.
//  2. RESOLVE: hit test through the page table (independent gathers), miss
//     compaction with prefix sums, victims from an explicit LRU list — slots
//     sorted by (stamp, slot).  A call only moves the slots it used to the most
//     recent end (they all get the newest stamp, so they sort by slot among
//     themselves), so two stable compactions maintain the list: no sort, no heap.
//     The evicted positions come from the prefetched reverse map, so eviction
//     issues stores only.
//  3. the host fetch of the missed rows.  With fetch_mode 1 this CTA copies them
//     from the mapped pinned host copy into their slots (serial, as the pages
//     describe).  With fetch_mode 0 it marks them in slot_of_sel and the attention
//     kernel copies them from host memory into its stage (and from there into
//     the slot) while the rest of the rows stream from HBM, so host-link time
//     overlaps HBM time.  fetch_mode 2 chooses per request: this kernel pulls
//     them all when the request's misses spread over the attention grid exceed a
//     few rows per CTA; otherwise it pulls only those in each attention CTA's
//     first units (needed at once) and leaves the rest, already moving into L2,
//     to the attention kernel.  All give identical results.  Either way every missed
//     row is prefetched into L2 (per 128-byte line) the moment its page lookup
//     misses, so the link starts working before the copies are issued.
//  4. the appended token: its index key to the HBM store, its K/V row to the
//     pinned host copy, length + 1 (stores that drain while the kernel ends).
#include "hs_internal.cuh"

namespace hs {

namespace {

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int FAST_MAX_N = 256 * 1024;   // one-pass top-k: contexts up to this many positions
constexpr int RES_WARPS = RES_THREADS / 32;
constexpr int WCAP = 256;                // digit-b1 keys a warp lists in the one-pass top-k
constexpr int AUTO_PULL_ROWS_PER_CTA = 8;  // fetch mode 2: pull here above this many misses per attention CTA
constexpr int FRONT_UNITS = 3;             // fetch mode 2: misses in an attention CTA's first units are pulled here
constexpr int CAND_MAX_N_PER_K = 20;       // candidate listing only for contexts up to 20 k positions
constexpr size_t SMEM_LIMIT = 227 * 1024;

struct ResLayout {
  size_t hist, sel, slot, miss_i, victim, ord, rev, used, bitmap, lists, newrow, total;
  bool rev_smem, fast;
};

__host__ __device__ inline ResLayout res_layout(const Geometry& g) {
  const int B = g.hot_slots, K = g.top_k;
  ResLayout L;
  size_t off = 0;
  L.hist = off;
  off += IDX_BINS * 4;
  L.sel = off;
  off += align_up((size_t)K * 4, 16);
  L.slot = off;
  off += align_up((size_t)K * 4, 16);
  L.miss_i = off;
  off += align_up((size_t)K * 4, 16);
  L.victim = off;
  off += align_up((size_t)K * 4, 16);
  L.ord = off;
  off += (size_t)B * 4;
  L.used = off;
  off += align_up((size_t)B, 16);
  L.newrow = off;
  off += align_up((size_t)g.row_bytes, 16) + align_up((size_t)g.d_idx, 16);
  const size_t base = off;
  // optional parts, in order of value: the one-pass top-k, then the reverse map
  const size_t fast_bytes = (size_t)FAST_MAX_N / 8 + (size_t)WCAP * RES_WARPS * 4;
  L.fast = base + fast_bytes <= SMEM_LIMIT;
  L.bitmap = off;
  if (L.fast) off += (size_t)FAST_MAX_N / 8;
  L.lists = off;
  if (L.fast) off += (size_t)WCAP * RES_WARPS * 4;
  L.rev = off;
  L.rev_smem = off + (size_t)B * 4 <= SMEM_LIMIT;
  if (L.rev_smem) off += (size_t)B * 4;
  L.total = off;
  return L;
}

struct ResShared {
  int scan[2 * (RES_THREADS / 32 + 1)];
  int b1, above1, b2, above2, bt, above_t;
  int rb1, rabove1, rb2, rabove2;   // random replacement: digits of the m-th smallest key
  int N, len, t_step, cnt;
  uint32_t thr;
};

// Finds the digit holding the kneed-th largest key (bins scanned from the top)
// and the number of keys in higher digits.
__device__ __forceinline__ void select_digit(const uint32_t* h, int kneed, int* scan, int* out_b,
                                             int* out_above) {
  constexpr int PER = IDX_BINS / RES_THREADS;   // bins per thread, descending
  const int tid = threadIdx.x;
  const int top = IDX_BINS - 1 - tid * PER;
  int v = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) v += (int)h[top - j];
  int tot;
  const int ex = block_exclusive_scan<RES_THREADS>(v, scan, &tot);
  if (ex < kneed && kneed <= ex + v) {
    int acc = ex;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int hv = (int)h[top - j];
      if (acc < kneed && kneed <= acc + hv) {
        *out_b = top - j;
        *out_above = acc;
      }
      acc += hv;
    }
  }
  __syncthreads();
}

// Random replacement's rank of an unpinned slot as a 24-bit value, larger =
// evicted first (the digit selection scans from the top): never-filled slots
// 0xFFFFFF (they go first, lowest slot first, as under LRU); a filled slot
// 0x7FFFFF minus the top 23 bits of SplitMix64 (Steele, Lea and Flood, "Fast
// splittable pseudorandom number generators", 2014; the finaliser constants of
// Vigna's reference code) for draw number counter + 1 from state seed, with
// counter = ((request * n_layers + layer) << 40) | ((step mod 2^24) << 16) | slot.
__device__ __forceinline__ uint32_t random_ikey(unsigned long long seed, unsigned long long rl, int step, int slot,
                                                bool empty) {
  if (empty) return 0xFFFFFFu;
  const unsigned long long ctr = (rl << 40) | ((unsigned long long)(step & 0xFFFFFF) << 16) | (unsigned)slot;
  unsigned long long z = seed + (ctr + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return 0x7FFFFFu - (uint32_t)(z >> 41);
}

}  // namespace

size_t resolve_smem_bytes(const Geometry& g) { return res_layout(g).total; }

__global__ void __launch_bounds__(RES_THREADS, 1) topk_resolve_kernel(DecodeParams p) {
  const Geometry& g = p.g;
  const int tid = threadIdx.x;
  const int ri = blockIdx.x;
  const int K = g.top_k;
  const int B = g.hot_slots;

  extern __shared__ __align__(16) unsigned char smem_raw[];
  const ResLayout L = res_layout(g);
  __shared__ ResShared sh;
  uint32_t* h = reinterpret_cast<uint32_t*>(smem_raw + L.hist);
  int32_t* sel = reinterpret_cast<int32_t*>(smem_raw + L.sel);
  int32_t* slot_sel = reinterpret_cast<int32_t*>(smem_raw + L.slot);
  int32_t* miss_i = reinterpret_cast<int32_t*>(smem_raw + L.miss_i);
  int32_t* victim = reinterpret_cast<int32_t*>(smem_raw + L.victim);
  int32_t* ord = reinterpret_cast<int32_t*>(smem_raw + L.ord);
  int32_t* rev_s = reinterpret_cast<int32_t*>(smem_raw + L.rev);
  uint8_t* used = smem_raw + L.used;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem_raw + L.bitmap);
  uint32_t* lists = reinterpret_cast<uint32_t*>(smem_raw + L.lists);   // [warp][WCAP]
  unsigned char* newrow = smem_raw + L.newrow;
  unsigned char* newkey = newrow + align_up((size_t)g.row_bytes, 16);
  HS_TRACE(p, 1, 0);

  for (int j = tid; j < B; j += RES_THREADS) used[j] = 0;
  griddep_wait();   // the score kernel's keys and histogram, earlier appends
  griddep_launch_dependents();

  int32_t* sel_g = p.s.sel + (long long)ri * K;
  int32_t* sel_out = p.sel_out ? p.sel_out + (long long)ri * K : nullptr;
  const int req = p.req_ids ? p.req_ids[ri] : ri;
  if (req < 0 || req >= g.max_requests) {
    if (tid == 0) set_error(p.s.dev_error, HS_DEVERR_REQ_RANGE);
    if (sel_out)
      for (int i = tid; i < K; i += RES_THREADS) sel_out[i] = -1;
    return;
  }
  const long long rl = (long long)req * g.n_layers + p.layer;

  // ---- 0. every read the chain needs, issued together ----------------------------
  const int32_t* order_g = p.s.order + rl * B;
  for (int c4 = tid; c4 < B / 4; c4 += RES_THREADS) cp_async_16(ord + 4 * c4, order_g + 4 * c4);
  if (L.rev_smem) {
    const int32_t* rev_g = p.s.reverse + rl * B;
    for (int c4 = tid; c4 < B / 4; c4 += RES_THREADS) cp_async_16(rev_s + 4 * c4, rev_g + 4 * c4);
  }
  uint32_t* gh = p.s.hist + (long long)ri * IDX_BINS;
  static_assert(IDX_BINS == 4 * RES_THREADS, "one 16-byte histogram chunk per thread");
  cp_async_16(h + 4 * tid, gh + 4 * tid);
  if (p.new_kv) {
    for (int v = tid; v < g.row_bytes / 16; v += RES_THREADS)
      cp_async_16(newrow + 16 * v, reinterpret_cast<const unsigned char*>(p.new_kv + (long long)ri * g.row_elems) + 16 * v);
    if (tid < g.d_idx / 16) cp_async_16(newkey + 16 * tid, p.new_keys + (long long)ri * g.d_idx + 16 * tid);
  }
  if (tid == 0) {
    const int len = p.s.length[rl];
    sh.len = len;
    sh.t_step = p.s.step[rl];
    sh.thr = p.s.cand_thr[rl];
    sh.cnt = (int)min(p.s.cand_cnt[ri], 0x7fffffffu);
    p.s.cand_cnt[ri] = 0;   // ready for the next call
    int N = len;
    if (p.new_kv) {
      if (len + 1 <= g.max_context) N = len + 1;
      else set_error(p.s.dev_error, HS_DEVERR_CAPACITY);
    }
    sh.N = N;
  }
  cp_async_wait_all();
  __syncthreads();
  const int len = sh.len, N = sh.N, t_step = sh.t_step;
  const bool appended = N > len;
  const int kk = min(K, N);
  HS_TRACE(p, 1, 1);

  // ======================= 1. top-k, ascending =======================
  if (N <= K) {
    for (int i = tid; i < N; i += RES_THREADS) sel[i] = i;
    if (tid == 0) p.s.cand_thr[rl] = 0u;
  } else {
    const uint32_t* keys = p.s.scores + (long long)ri * p.score_stride;
    reinterpret_cast<uint4*>(gh)[tid] = make_uint4(0, 0, 0, 0);   // ready for the next call
    // the digit of the k-th largest key, and the digit above which ~1.25 k keys lie:
    // the next call lists keys from there on (exact whenever >= k of them clear it)
    const int k_next = (int)min((long long)N, (long long)K + K / 4);
    select_digit(h, K, sh.scan, &sh.b1, &sh.above1);
    select_digit(h, k_next, sh.scan, &sh.bt, &sh.above_t);
    const int b1 = sh.b1, above1 = sh.above1;
    // listing costs the score kernel about as much per position as the full pass
    // costs here, so it pays only while the context is short relative to k
    if (tid == 0) p.s.cand_thr[rl] = N <= CAND_MAX_N_PER_K * K ? (uint32_t)sh.bt << 12 : 0u;
    reinterpret_cast<uint4*>(h)[tid] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    HS_TRACE(p, 1, 2);
    // each thread: a contiguous range of whole 32-position words
    // per-thread contiguous ranges (the rescan path)
    const int per = ((N + RES_THREADS - 1) / RES_THREADS + 3) & ~3;
    const int j0 = min(N, tid * per), j1 = min(N, j0 + per);
    // per-warp contiguous chunks of 128 positions (the one-pass path)
    const int lane = tid & 31, wid = tid >> 5;
    const int NC = (N + 127) >> 7;
    const int c0 = (int)((long long)wid * NC / RES_WARPS), c1 = (int)((long long)(wid + 1) * NC / RES_WARPS);
    uint32_t* wl = lists + wid * WCAP;
    const int cap = 2 * K;
    const bool use_cand = L.fast && N <= FAST_MAX_N && sh.thr != 0u && sh.cnt >= K && sh.cnt <= cap;
    const bool fast = !use_cand && L.fast && N <= FAST_MAX_N;
    int wcnt = 0;       // entries of this warp's list (warp-uniform)
    int lane_gt = 0;    // keys above digit b1 seen by this lane
    bool overflow = false;
    const uint2* cl = p.s.cand + (long long)ri * cap;   // this call's candidates
    uint32_t* tiebm = lists;                            // the candidate path's second bitmap
    const int NW = (N + 31) >> 5;
    if (use_cand) {
      // every key >= the threshold is listed and at least k are: the k largest
      // (ties included) are all in the list.  Second digit from the list only.
      for (int q = tid; q < NW; q += RES_THREADS) {
        bitmap[q] = 0u;
        tiebm[q] = 0u;
      }
      const int32_t* page_rl = p.s.page + rl * g.max_context;
      for (int i = tid; i < sh.cnt; i += RES_THREADS) {
        const uint2 c = __ldcg(&cl[i]);
        if ((int)(c.y >> 12) == b1) atomicAdd(&h[c.y & 4095u], 1u);
        // every selected position is a candidate: warm its page-table entry for the hit test
        asm volatile("prefetch.global.L2 [%0];" ::"l"(page_rl + c.x));
      }
    } else if (fast) {
      const uint4* k4 = reinterpret_cast<const uint4*>(keys);   // rows padded to a multiple of 4 keys
      constexpr int UC = 8;   // chunks in flight per lane (a 32K-position row in one round)
      for (int cb = c0; cb < c1; cb += UC) {
        uint4 v[UC];
#pragma unroll
        for (int u = 0; u < UC; ++u) {
          const int pos = 128 * (cb + u) + 4 * lane;
          v[u] = (cb + u < c1 && pos < N) ? k4[(cb + u) * 32 + lane] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < UC; ++u) {
          if (cb + u >= c1) break;   // warp-uniform
          const int pos = 128 * (cb + u) + 4 * lane;
          const uint32_t kv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          uint32_t nib_gt = 0, nib_eq = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (pos + e < N) {
              const int dg = (int)(kv[e] >> 12);
              nib_gt |= (uint32_t)(dg > b1) << e;
              if (dg == b1) {
                nib_eq |= 1u << e;
                atomicAdd(&h[kv[e] & 4095u], 1u);
              }
            }
          }
          lane_gt += __popc(nib_gt);
          uint32_t word = nib_gt << (4 * (lane & 7));
          word |= __shfl_xor_sync(FULL_MASK, word, 1);
          word |= __shfl_xor_sync(FULL_MASK, word, 2);
          word |= __shfl_xor_sync(FULL_MASK, word, 4);
          if ((lane & 7) == 0) bitmap[4 * (cb + u) + (lane >> 3)] = word;
          if (__any_sync(FULL_MASK, nib_eq != 0)) {   // list the digit-b1 keys in position order
            const int cnt = __popc(nib_eq);
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int n = __shfl_up_sync(FULL_MASK, incl, o);
              if (lane >= o) incl += n;
            }
            int at = wcnt + incl - cnt;
            for (int e = 0; e < 4; ++e)
              if ((nib_eq >> e) & 1u) {
                if (at < WCAP) wl[at] = ((uint32_t)(pos + e) << 12) | (kv[e] & 4095u);
                else overflow = true;
                ++at;
              }
            wcnt += __shfl_sync(FULL_MASK, incl, 31);
          }
        }
      }
    } else {   // second-digit histogram only; the counts and the emission rescan the keys
      const int n4 = N >> 2;
      const uint4* k4 = reinterpret_cast<const uint4*>(keys);
      constexpr int UA = 8;   // loads in flight per thread
      for (int i0 = tid; i0 < n4; i0 += UA * RES_THREADS) {
        uint4 v[UA];
#pragma unroll
        for (int u = 0; u < UA; ++u) {
          const int i = i0 + u * RES_THREADS;
          v[u] = i < n4 ? k4[i] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < UA; ++u) {
          if ((int)(v[u].x >> 12) == b1) atomicAdd(&h[v[u].x & 4095u], 1u);
          if ((int)(v[u].y >> 12) == b1) atomicAdd(&h[v[u].y & 4095u], 1u);
          if ((int)(v[u].z >> 12) == b1) atomicAdd(&h[v[u].z & 4095u], 1u);
          if ((int)(v[u].w >> 12) == b1) atomicAdd(&h[v[u].w & 4095u], 1u);
        }
      }
      for (int i = 4 * n4 + tid; i < N; i += RES_THREADS) {
        const uint32_t v = keys[i];
        if ((int)(v >> 12) == b1) atomicAdd(&h[v & 4095u], 1u);
      }
    }
    // the barrier is taken on every path (it orders the histogram atomics above
    // before the digit select below), then decides whether the lists are usable
    const bool any_overflow = __syncthreads_or(overflow);
    const bool use_lists = fast && !any_overflow;
    HS_TRACE(p, 1, 3);
    select_digit(h, K - above1, sh.scan, &sh.b2, &sh.above2);
    HS_TRACE(p, 1, 4);
    const int b2 = sh.b2;
    const uint32_t vstar = ((uint32_t)b1 << 12) | (uint32_t)b2;
    const int need_eq = K - (above1 + sh.above2);   // >= 1
    if (use_cand) {
      // mark the taken keys (> threshold) and the threshold ties in two bitmaps
      for (int i = tid; i < sh.cnt; i += RES_THREADS) {
        const uint2 c = __ldcg(&cl[i]);
        if (c.y > vstar) atomicOr(&bitmap[c.x >> 5], 1u << (c.x & 31));
        else if (c.y == vstar) atomicOr(&tiebm[c.x >> 5], 1u << (c.x & 31));
      }
      __syncthreads();
      // per-warp word ranges, counts, scan over the warps
      const int q0w = (int)((long long)wid * NW / RES_WARPS), q1w = (int)((long long)(wid + 1) * NW / RES_WARPS);
      int n_gt = 0, n_eq = 0;
      for (int q = q0w + lane; q < q1w; q += 32) {
        n_gt += __popc(bitmap[q]);
        n_eq += __popc(tiebm[q]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        n_gt += __shfl_xor_sync(FULL_MASK, n_gt, o);
        n_eq += __shfl_xor_sync(FULL_MASK, n_eq, o);
      }
      const int2 wb = block_exclusive_scan2<RES_THREADS>(lane == 0 ? n_gt : 0, lane == 0 ? n_eq : 0, sh.scan,
                                                         nullptr, nullptr);
      const int gt_before = __shfl_sync(FULL_MASK, wb.x, 0), eq_before = __shfl_sync(FULL_MASK, wb.y, 0);
      HS_TRACE(p, 1, 5);
      int out = gt_before + min(eq_before, need_eq);
      int tie_run = eq_before;   // threshold ties before this group of words
      for (int qg = q0w; qg < q1w; qg += 32) {
        const int q = qg + lane;
        uint32_t m = q < q1w ? bitmap[q] : 0u;
        uint32_t tb = q < q1w ? tiebm[q] : 0u;
        const int nt = __popc(tb);
        int tincl = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(FULL_MASK, tincl, o);
          if (lane >= o) tincl += n;
        }
        int rank = tie_run + tincl - nt;   // ties take the lowest positions first
        while (tb) {
          const int bb = __ffs(tb) - 1;
          tb &= tb - 1;
          if (rank < need_eq) m |= 1u << bb;
          ++rank;
        }
        tie_run += __shfl_sync(FULL_MASK, tincl, 31);
        const int cnt = __popc(m);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(FULL_MASK, incl, o);
          if (lane >= o) incl += n;
        }
        int o = out + incl - cnt;
        while (m) {
          const int bb = __ffs(m) - 1;
          m &= m - 1;
          if (o < K) sel[o++] = 32 * q + bb;
        }
        out += __shfl_sync(FULL_MASK, incl, 31);
      }
    } else if (use_lists) {
      // per-warp counts, then a scan over the warps
      int n_gt = lane_gt, n_eq = 0;
      for (int q = lane; q < wcnt; q += 32) {
        const int lo = (int)(wl[q] & 4095u);
        n_gt += lo > b2;
        n_eq += lo == b2;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        n_gt += __shfl_xor_sync(FULL_MASK, n_gt, o);
        n_eq += __shfl_xor_sync(FULL_MASK, n_eq, o);
      }
      const int2 wb = block_exclusive_scan2<RES_THREADS>(lane == 0 ? n_gt : 0, lane == 0 ? n_eq : 0, sh.scan,
                                                         nullptr, nullptr);
      const int gt_before = __shfl_sync(FULL_MASK, wb.x, 0), eq_before = __shfl_sync(FULL_MASK, wb.y, 0);
      HS_TRACE(p, 1, 5);
      // emission: lane l owns bitmap word q0 + l of each group of 32 words
      int out = gt_before + min(eq_before, need_eq);
      int tie_run = eq_before;   // ties before the current list entry (position order)
      int qe = 0;                // next list entry
      const int w_end = 4 * c1;
      for (int q0 = 4 * c0; q0 < w_end; q0 += 32) {
        const int q = q0 + lane;
        uint32_t m = q < w_end ? bitmap[q] : 0u;
        for (; qe < wcnt; ++qe) {   // list entries of this group of words, in order
          const uint32_t e = wl[qe];
          const int pos = (int)(e >> 12);
          if ((pos >> 5) >= q0 + 32) break;
          const int lo = (int)(e & 4095u);
          const bool mine = (pos >> 5) == q;
          if (lo > b2) {
            if (mine) m |= 1u << (pos & 31);
          } else if (lo == b2) {
            if (mine && tie_run < need_eq) m |= 1u << (pos & 31);
            ++tie_run;
          }
        }
        const int cnt = __popc(m);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(FULL_MASK, incl, o);
          if (lane >= o) incl += n;
        }
        int o = out + incl - cnt;
        while (m) {
          const int bb = __ffs(m) - 1;
          m &= m - 1;
          if (o < K) sel[o++] = 32 * q + bb;
        }
        out += __shfl_sync(FULL_MASK, incl, 31);
      }
    } else {
      int n_gt = 0, n_eq = 0;
      for (int j = j0; j < j1; j += 4) {   // multiples of 4 in bounds (padded rows)
        const uint4 v = *reinterpret_cast<const uint4*>(keys + j);
        const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (j + e < j1) {
            n_gt += kv[e] > vstar;
            n_eq += kv[e] == vstar;
          }
      }
      const int2 before = block_exclusive_scan2<RES_THREADS>(n_gt, n_eq, sh.scan, nullptr, nullptr);
      HS_TRACE(p, 1, 5);
      int o = before.x + min(before.y, need_eq);
      int eq_rank = before.y;
      for (int j = j0; j < j1; j += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + j);
        const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (j + e < j1) {
            bool take = kv[e] > vstar;
            if (kv[e] == vstar) {
              take = eq_rank < need_eq;
              ++eq_rank;
            }
            if (take && o < K) sel[o++] = j + e;
          }
      }
    }
  }
  __syncthreads();
  HS_TRACE(p, 1, 6);
  for (int i = tid; i < K; i += RES_THREADS) {
    const int v = i < kk ? sel[i] : -1;
    if (i < kk) sel_g[i] = v;
    if (sel_out) sel_out[i] = v;
  }

  // ======================= 2. RESOLVE metadata =======================
  int32_t* page = p.s.page + rl * g.max_context;
  int32_t* reverse = p.s.reverse + rl * B;
  int32_t* stamp = p.s.stamp + rl * B;
  int32_t* order = p.s.order + rl * B;
  const int t = t_step;
  int m = 0;
  bool pull = false, front_pull = false;   // who copies this request's missed rows (see below)
  if (kk > 0) {
    // hit test: independent page-table gathers, four in flight per thread
    bool bad = false;
    for (int i0 = tid; i0 < kk; i0 += 4 * RES_THREADS) {
      int pos[4], s4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * RES_THREADS;
        pos[u] = i < kk ? sel[i] : -1;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) s4[u] = (pos[u] >= 0 && pos[u] < N) ? page[pos[u]] : -1;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * RES_THREADS;
        if (i < kk) {
          if (pos[u] < 0 || pos[u] >= N || s4[u] >= B) bad = true;
          slot_sel[i] = s4[u];
          if (s4[u] >= 0 && s4[u] < B) used[s4[u]] = 1;
          // a miss: start moving its host row over the link into L2 now, line by
          // line (the pull below, or the attention kernel in fetch mode 0, then
          // reads it from L2); the row appended by this call is written below
          if (s4[u] < 0 && pos[u] >= 0 && pos[u] < N && !(appended && pos[u] == len)) {
            const unsigned char* src = reinterpret_cast<const unsigned char*>(p.s.host_kv) +
                                       ((size_t)rl * g.max_context + pos[u]) * g.row_bytes;
            for (int b = 0; b < g.row_bytes; b += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + b));
          }
        }
      }
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) set_error(p.s.dev_error, HS_DEVERR_METADATA);
      return;   // slot_of_sel keeps in-range values from before: the attention stays in bounds
    }
    HS_TRACE(p, 1, 7);
    // misses in ascending selection order, and the unpinned entries of the LRU list
    const int per_i = (kk + RES_THREADS - 1) / RES_THREADS;
    const int i0 = min(kk, tid * per_i), i1 = min(kk, i0 + per_i);
    const int per_j = (B + RES_THREADS - 1) / RES_THREADS;
    const int j0 = min(B, tid * per_j), j1 = min(B, j0 + per_j);
    int nm = 0, nc = 0;
    for (int i = i0; i < i1; ++i) nm += slot_sel[i] < 0;
    for (int j = j0; j < j1; ++j) nc += used[ord[j]] == 0;
    HS_TRACE(p, 1, 20);
    const int2 mc = block_exclusive_scan2<RES_THREADS>(nm, nc, sh.scan, &m, nullptr);
    HS_TRACE(p, 1, 21);
    int mb = mc.x;
    for (int i = i0; i < i1; ++i)
      if (slot_sel[i] < 0) miss_i[mb++] = i;
    if (p.replacement == HS_REPLACE_RANDOM) {
      // victims: the m unpinned slots ranked first (never-filled, then smallest
      // (key, slot)), in ascending slot order.  Two 12-bit digit selections over
      // the 24-bit ranks (the same histogram scan as the top-k), then each thread
      // takes its ranks above the threshold and, in slot order, the threshold ties
      // still needed.  Slots are visited by index (this thread's range j0..j1);
      // "never filled" is read from the reverse map as it was before this call.
      if (m > 0) {
        const unsigned long long seed = p.replacement_seed;
        auto rank_of = [&](int j) {
          const int old = L.rev_smem ? rev_s[j] : reverse[j];
          return random_ikey(seed, rl, t, j, old < 0);
        };
        reinterpret_cast<uint4*>(h)[tid] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        for (int j = j0; j < j1; ++j)
          if (used[j] == 0) atomicAdd(&h[rank_of(j) >> 12], 1u);
        __syncthreads();
        select_digit(h, m, sh.scan, &sh.rb1, &sh.rabove1);
        const int rb1 = sh.rb1, rab1 = sh.rabove1;
        reinterpret_cast<uint4*>(h)[tid] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        for (int j = j0; j < j1; ++j)
          if (used[j] == 0) {
            const uint32_t k = rank_of(j);
            if ((int)(k >> 12) == rb1) atomicAdd(&h[k & 4095u], 1u);
          }
        __syncthreads();
        select_digit(h, m - rab1, sh.scan, &sh.rb2, &sh.rabove2);
        const uint32_t vstar = ((uint32_t)rb1 << 12) | (uint32_t)sh.rb2;
        const int need_eq = m - rab1 - sh.rabove2;   // >= 1
        int n_gt = 0, n_eq = 0;
        for (int j = j0; j < j1; ++j)
          if (used[j] == 0) {
            const uint32_t k = rank_of(j);
            n_gt += k > vstar;
            n_eq += k == vstar;
          }
        const int2 ex = block_exclusive_scan2<RES_THREADS>(n_gt, n_eq, sh.scan, nullptr, nullptr);
        int eq_rank = ex.y;                        // threshold ties before this thread
        int o = ex.x + min(ex.y, need_eq);         // victims before this thread
        for (int j = j0; j < j1; ++j)
          if (used[j] == 0) {
            const uint32_t k = rank_of(j);
            const bool take = k > vstar || (k == vstar && eq_rank++ < need_eq);
            if (take) {
              victim[o++] = j;
              used[j] = 2;
            }
          }
      }
    } else {
      // victims: the first m unpinned entries of the (stamp, slot)-sorted list
      int cb = mc.y;
      for (int j = j0; j < j1 && cb < m; ++j) {
        const int sl = ord[j];
        if (used[sl] == 0) {
          victim[cb++] = sl;
          used[sl] = 2;
        }
      }
    }
    __syncthreads();
    HS_TRACE(p, 1, 8);
    // evict, then record the new residents (stores only)
    for (int q = tid; q < m; q += RES_THREADS) {
      const int v = victim[q];
      const int i = miss_i[q];
      const int pnew = sel[i];
      const int old = L.rev_smem ? rev_s[v] : reverse[v];
      if (old >= 0 && old < g.max_context) page[old] = -1;
      reverse[v] = pnew;
      page[pnew] = v;
      slot_sel[i] = v;
    }
    __syncthreads();
    HS_TRACE(p, 1, 9);
    // slot of every selected position (misses flagged for the attention kernel
    // when it does the fetch); stamp every used slot
    // who copies the missed rows: fetch mode 1 (or 2 with many misses per
    // attention CTA) = this kernel below, else the attention kernel, which
    // overlaps a few rows per CTA with its HBM reads but stalls on many
    pull = p.fetch_mode == 1 ||
           (p.fetch_mode == 2 && (long long)m * p.n_req > (long long)AUTO_PULL_ROWS_PER_CTA * p.att_grid);
    // fetch mode 2 with few misses: the attention kernel copies them, except those
    // in the first FRONT_UNITS units of each attention CTA (needed before any
    // prefetch could land), which are pulled here.  The attention kernel splits
    // the flattened units of all requests into equal ranges over min(grid, U)
    // CTAs; the same split is recomputed from every request's k_eff.
    front_pull = p.fetch_mode == 2 && !pull && !g.shared_kv && p.s.call_n != nullptr;
    if (front_pull) {
      const int tile = ATT_SUBTILE * (8 / g.h_kv);
      int before = 0, all = 0;
      for (int j = tid; j < p.n_req; j += RES_THREADS) {
        const int u = (min(K, p.s.call_n[j]) + tile - 1) / tile;
        all += u;
        if (j < ri) before += u;
      }
      int t_before, t_all;
      (void)block_exclusive_scan2<RES_THREADS>(before, all, sh.scan, &t_before, &t_all);
      const long long U = t_all;
      const int Gc = (int)max(1LL, min((long long)p.att_grid, U));
      for (int q = tid; q < m; q += RES_THREADS) {
        const long long u = t_before + miss_i[q] / tile;
        const long long c = ((u + 1) * Gc + U - 1) / U - 1;   // owning attention CTA
        const bool front = u - c * U / Gc < FRONT_UNITS;
        miss_i[q] = front ? (miss_i[q] | HS_SLOT_MISS_FLAG) : miss_i[q];   // mark: pulled here
      }
      __syncthreads();
    }
    auto pulled = [&](int q) { return pull || (front_pull && (miss_i[q] & HS_SLOT_MISS_FLAG)); };
    auto miss_sel = [&](int q) { return miss_i[q] & ~HS_SLOT_MISS_FLAG; };
    const int miss_flag = pull ? 0 : HS_SLOT_MISS_FLAG;
    int32_t* sos = p.s.slot_of_sel + (long long)ri * K;
    // LRU and random: every used slot is refreshed; FIFO: only the filled ones (used == 2)
    const bool fifo = p.replacement == HS_REPLACE_FIFO;
    auto refreshed = [&](uint8_t u) { return fifo ? u == 2 : u != 0; };
    for (int i = tid; i < kk; i += RES_THREADS) {
      const int sl = slot_sel[i];
      if (refreshed(used[sl])) stamp[sl] = t;
      sos[i] = sl;
    }
    HS_TRACE(p, 1, 22);
    __syncthreads();
    HS_TRACE(p, 1, 23);
    for (int q = tid; q < m; q += RES_THREADS) sos[miss_sel(q)] = victim[q] | (pulled(q) ? 0 : miss_flag);
    // new list: slots not refreshed keep their order, refreshed slots (all with
    // the newest stamp) go last by slot
    int nu = 0, nus = 0;
    for (int j = j0; j < j1; ++j) nu += !refreshed(used[ord[j]]);
    for (int sl = j0; sl < j1; ++sl) nus += refreshed(used[sl]);
    int n_unused;
    HS_TRACE(p, 1, 24);
    const int2 un = block_exclusive_scan2<RES_THREADS>(nu, nus, sh.scan, &n_unused, nullptr);
    HS_TRACE(p, 1, 25);
    int ub = un.x;
    for (int j = j0; j < j1; ++j) {
      const int sl = ord[j];
      if (!refreshed(used[sl])) order[ub++] = sl;
    }
    int sb = n_unused + un.y;
    for (int sl = j0; sl < j1; ++sl)
      if (refreshed(used[sl])) order[sb++] = sl;
    HS_TRACE(p, 1, 26);
    if (tid == 0) {
      p.s.step[rl] = t + 1;
      red_add_u64(&p.s.hits[rl], (unsigned long long)(kk - m));
      red_add_u64(&p.s.misses[rl], (unsigned long long)m);
      red_add_u64(&p.s.glob[0], (unsigned long long)m * g.row_bytes);
    }
    HS_TRACE(p, 1, 10);
  }

  // ======================= 4. the appended token =======================
  if (appended) {
    const int rvec = g.row_bytes / 16;
    int4* dst = reinterpret_cast<int4*>(p.s.host_kv + (rl * g.max_context + len) * g.row_elems);
    for (int v = tid; v < rvec; v += RES_THREADS) dst[v] = reinterpret_cast<const int4*>(newrow)[v];
    if (tid < g.d_idx / 16)
      reinterpret_cast<int4*>(p.s.idx_keys + (rl * g.max_context + len) * g.d_idx)[tid] =
          reinterpret_cast<const int4*>(newkey)[tid];
    if (tid == 0) {
      p.s.length[rl] = N;
      red_add_u64(&p.s.glob[1], (unsigned long long)g.row_bytes);
    }
  }

  // ======================= 3. host fetch (fetch_mode 1) =======================
  if (m > 0 && (pull || front_pull)) {
    const int rvec = g.row_bytes / 16;
    const long long total = (long long)m * rvec;
    const unsigned char* src_base =
        reinterpret_cast<const unsigned char*>(p.s.host_kv) + (size_t)rl * g.max_context * g.row_bytes;
    unsigned char* dst_base = reinterpret_cast<unsigned char*>(p.s.hot) + (size_t)rl * B * g.row_bytes;
    constexpr int U = 8;   // 128 KB of host reads in flight per CTA
    for (long long e0 = tid; e0 < total; e0 += (long long)U * RES_THREADS) {
      int4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long e = e0 + (long long)u * RES_THREADS;
        const int q = e < total ? (int)(e / rvec) : 0;
        if (e < total && (pull || (miss_i[q] & HS_SLOT_MISS_FLAG))) {
          const int cidx = (int)(e - (long long)q * rvec);
          const int pos = sel[miss_i[q] & ~HS_SLOT_MISS_FLAG];
          // the token appended by this call is read from its input copy
          v[u] = (appended && pos == len) ? reinterpret_cast<const int4*>(newrow)[cidx]
                                          : *reinterpret_cast<const int4*>(src_base + (size_t)pos * g.row_bytes + cidx * 16);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long e = e0 + (long long)u * RES_THREADS;
        const int q = e < total ? (int)(e / rvec) : 0;
        if (e < total && (pull || (miss_i[q] & HS_SLOT_MISS_FLAG))) {
          const int cidx = (int)(e - (long long)q * rvec);
          *reinterpret_cast<int4*>(dst_base + (size_t)victim[q] * g.row_bytes + cidx * 16) = v[u];
        }
      }
    }
  }
  HS_TRACE(p, 1, 13);
}

// An ordinary launch, not a programmatic dependent of the score kernel: launched
// early, these CTAs would take the SMs the score kernel's CTAs free first, and
// with many host rows to pull that placement cost up to half the link rate
// (measured: 1.65 against 1.16 ms per layer-step at 29 % misses).  Launched
// after the score kernel completes, the scheduler spreads them over the GPU.
// The kernel's own griddepcontrol.wait then returns at once, and it still lets
// the attention kernel launch early.
cudaError_t launch_resolve(const DecodeParams& p, size_t smem, cudaStream_t st) {
  topk_resolve_kernel<<<p.n_req, RES_THREADS, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t prepare_resolve(size_t smem) {
  return allow_smem(topk_resolve_kernel, smem);
}

}  // namespace hs
