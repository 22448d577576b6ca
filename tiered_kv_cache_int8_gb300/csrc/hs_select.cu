// The select kernel: indexer scores, exact top-k and RESOLVE of one decode
// layer-step for every request, in ONE persistent launch, so that a request's
// selection and cache update start as soon as its own scores exist instead of
// after every request has been scored.
//
// Method.  "10月14日学习笔记" (zgchen.com), "HiSparse / 动机": an indexer scores
// the context and attention runs over the top-k positions (ties here: the lower
// position; output ascending).  The score is an int8 query dotted with each
// position's int8 index key, summed exactly in int32 with dp4a.
// "KV卸载上主机:HiSparse、PDD与DDR4回收", "论文1：HiSparse": a page table plus
// LRU metadata drive replacement of the B hot slots of each (request, layer);
// hit detection, LRU replacement, metadata update and the host fetch are
// resolved in one kernel per layer.  "10月14日学习笔记", "方法" 1: adjacent
// steps overlap, so LRU fits.
//
// Replacement rule: slots holding a selected position (hits) are pinned; the m
// misses, in ascending position order, go to the m unpinned slots with the
// smallest (stamp, slot), in that order; every used slot's stamp (LRU), or only
// every filled slot's (FIFO, a comparison policy of the pages), becomes the
// (request, layer) step counter, which then grows by one.  Random replacement
// (the other comparison policy) takes the m unpinned slots with the smallest
// counter-based hash keys instead, in ascending slot order, and stamps as LRU.
//
// Design (sm_103a).  Grid = one 512-thread CTA per SM.  CTAs 0..n_resolvers-1
// are resolvers, the rest score:
//  * Scoring is HBM-bound (d_idx bytes per position).  The positions of every
//    request that needs a selection (more positions than k) are flattened in
//    request order and cut into warp tiles (two sub-tiles of 8 x 16-byte loads
//    per lane); scorer warp w takes tiles w, w + W, w + 2W, ... so all warps
//    sweep the requests in order and request r is complete early.  The DRAM
//    stream is driven by bulk L2 prefetches two rounds of tiles ahead (before
//    the grid dependency resolves, each warp already loads its first tile and
//    sends its second towards L2: the keys are the library's own); the tile is
//    read with coalesced 16-byte loads (the 8 lanes of a position read its
//    8 chunks side by side) that then hit L2, issued only after the previous
//    tile's release so that its fence does not wait for them; dp4a partial
//    sums are combined with lane shuffles.  Each key
//    (score + 2^22, order-preserving, 24 bits) goes to a scratch row; keys at or
//    above the request's candidate threshold (left by the previous call) are
//    also listed with their positions (one atomic per warp tile).  After a
//    tile its warp adds 1 to the request's tile counter with release order.
//  * A resolver takes requests j, j + n_resolvers, ...: it first prefetches
//    what does not depend on the scores (LRU list, reverse map, the appended
//    row), waits (bounded) until the request's tiles are all counted, then runs
//    the latency-bound chain:
//     - exact top-k: when the previous call's threshold listed between k and 2k
//       keys, the k largest (ties included) are all in the list, so a two-digit
//       radix select over the list alone finds them; otherwise a histogram pass
//       and one pass that turns "digit above the threshold digit" into a
//       position bitmap (the few keys with the threshold digit go to per-warp
//       lists in position order) over the scratch keys.  Either way the
//       selection is emitted ascending from bitmaps.
//     - RESOLVE: hit test through the page table (on the candidate path the page
//       entries come with the candidates, read by the scorers; else independent
//       gathers), miss compaction by warp segments (ballots, one block scan),
//       victims from an explicit LRU list kept
//       sorted by (stamp, slot) — a call moves exactly the slots it used to the
//       most recent end, so two stable compactions maintain it: no sort, no heap.
//     - publication: selection, slot of every selected row (misses flagged for
//       the attention kernel, which copies them host -> stage -> slot), then the
//       request's ready flag = k_eff + 1 (release).  The attention kernel, launched
//       as a programmatic dependent, starts on the requests that are ready while
//       later ones are still being scored or resolved.
//     - after publication (the attention kernel's prefetcher warp starts the
//       missed host rows moving into L2): the next threshold, stamps, the new
//       LRU list, counters, step + 1 and the
//       appended token (its key to the HBM store, its row to the pinned host
//       copy, length + 1).  Lengths and thresholds are written only once every
//       CTA of the launch has read them (a grid-wide counter).
//  * fetch_mode 1 (and latent rows, which every head group reads) pulls the
//    missed rows into their slots inside the resolver before publication.
//  * Write-allocate (a variant; the pages leave open whether a new token enters
//    the hot cache): the token a call appends counts as used by the call — when
//    the selection does not take it, it is one more miss after the selection,
//    filled from its input row into the last victim and stamped like the rest.
#include "hs_internal.cuh"

namespace hs {

namespace {

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int NT = SEL_THREADS;
constexpr int NWARP = NT / 32;
constexpr int FAST_MAX_N = 256 * 1024;   // one-pass top-k: contexts up to this many positions
constexpr int WCAP = 256;                // threshold-digit keys a warp lists in the one-pass top-k
constexpr int CAND_MAX_N_PER_K = 128;    // candidate listing for contexts up to 128 k positions
constexpr int CAND_REG = 8;              // listed candidates a resolver thread holds in registers
constexpr size_t SMEM_LIMIT = 227 * 1024;

// Per-request tables of the launch (scorers) and the resolver's layout share the
// dynamic shared memory: a CTA is one or the other.
struct SelLayout {
  // scorer tables
  size_t t_prefix, t_req, t_n, t_thr, t_total;
  // resolver
  size_t hist, sel, slot, miss_i, victim, ord, rev, used, bitmap, lists, wpre, newrow, r_total;
  bool rev_smem, fast;
  size_t total;
};

__host__ __device__ inline SelLayout sel_layout(const Geometry& g) {
  const int B = g.hot_slots, K = g.top_k;
  SelLayout L;
  size_t off = 0;
  L.t_prefix = off;   // int [n+1]: first warp tile of request i
  off += align_up((size_t)(g.max_requests + 1) * 4, 16);
  L.t_req = off;      // int [n]: request id (-1: nothing to score)
  off += align_up((size_t)g.max_requests * 4, 16);
  L.t_n = off;        // int [n]: positions this call (with the appended token)
  off += align_up((size_t)g.max_requests * 4, 16);
  L.t_thr = off;      // u32 [n]: candidate threshold
  off += align_up((size_t)g.max_requests * 4, 16);
  L.t_total = off;

  off = 0;
  L.hist = off;
  off += IDX_BINS * 4;
  L.sel = off;
  off += align_up((size_t)(K + 1) * 4, 16);
  L.slot = off;
  off += align_up((size_t)(K + 1) * 4, 16);
  L.miss_i = off;
  off += align_up((size_t)(K + 1) * 4, 16);
  L.victim = off;
  off += align_up((size_t)(K + 1) * 4, 16);
  L.ord = off;
  off += (size_t)B * 4;
  L.used = off;
  off += align_up((size_t)B, 16);
  L.newrow = off;
  off += align_up((size_t)g.row_bytes, 16) + align_up((size_t)g.d_idx, 16);
  const size_t base = off;
  // optional parts, in order of value: the one-pass top-k, then the reverse map
  // two position bitmaps, the per-warp lists and 16-bit per-word prefix counts
  const size_t fast_bytes = (size_t)FAST_MAX_N / 4 + (size_t)WCAP * NWARP * 4 + (size_t)FAST_MAX_N / 32 * 4;
  L.fast = base + fast_bytes <= SMEM_LIMIT;
  L.bitmap = off;
  if (L.fast) off += (size_t)FAST_MAX_N / 4;
  L.lists = off;
  if (L.fast) off += (size_t)WCAP * NWARP * 4;
  L.wpre = off;
  if (L.fast) off += (size_t)FAST_MAX_N / 32 * 4;
  L.rev = off;
  L.rev_smem = off + (size_t)B * 4 <= SMEM_LIMIT;
  if (L.rev_smem) off += (size_t)B * 4;
  L.r_total = off;
  L.total = L.t_total > L.r_total ? L.t_total : L.r_total;
  return L;
}

struct SelShared {
  int scan[2 * (NWARP + 1)];
  int b1, above1, b2, above2, bt, above_t;
  int thr_src;   // where the next threshold's low digit is found: 0 none, 1 the candidate list, 2 all keys
  int rb1, rabove1, rb2, rabove2;   // random replacement: digits of the m-th smallest key
  int len, N, t_step, cnt, req, ok;
  int t_step_f, len_f;   // a follower layer's step counter and length
  uint32_t thr, thr_next;
};

// Finds the digit holding the kneed-th largest key (bins scanned from the top)
// and the number of keys in higher digits; with kneed2 > 0 the same for a second
// rank in the same scan.  Leaves an output untouched when the histogram holds
// fewer keys than its rank.
__device__ __forceinline__ void select_digit(const uint32_t* h, int kneed, int* scan, int* out_b, int* out_above,
                                             int kneed2 = 0, int* out_b2 = nullptr, int* out_above2 = nullptr) {
  constexpr int PER = IDX_BINS / NT;   // bins per thread, descending
  static_assert(PER % 4 == 0, "whole 16-byte groups of bins per thread");
  const int tid = threadIdx.x;
  const int top = IDX_BINS - 1 - tid * PER;
  // the thread's bins top - PER + 1 .. top, read as 16-byte vectors (a lane
  // stride of PER words would otherwise conflict on the shared-memory banks)
  uint32_t hb[PER];
#pragma unroll
  for (int c = 0; c < PER / 4; ++c) {
    const uint4 x = reinterpret_cast<const uint4*>(h + top - PER + 1)[c];
    hb[4 * c] = x.x;
    hb[4 * c + 1] = x.y;
    hb[4 * c + 2] = x.z;
    hb[4 * c + 3] = x.w;
  }
  int v = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) v += (int)hb[j];
  int tot;
  const int ex = block_exclusive_scan<NT>(v, scan, &tot);
  auto find = [&](int kn, int* ob, int* oa) {
    if (ex < kn && kn <= ex + v) {
      int acc = ex;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int hv = (int)hb[PER - 1 - j];   // bin top - j
        if (acc < kn && kn <= acc + hv) {
          *ob = top - j;
          *oa = acc;
        }
        acc += hv;
      }
    }
  };
  find(kneed, out_b, out_above);
  if (kneed2 > 0) find(kneed2, out_b2, out_above2);
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

__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Streaming 16-byte load (read once: evicted first from L1 and L2).
__device__ __forceinline__ int4 ld_stream(const void* p) { return __ldcs(reinterpret_cast<const int4*>(p)); }

// ---------------------------------------------------------------------------
// scoring geometry for d_idx = 16 * NCH bytes
// ---------------------------------------------------------------------------
template <int NCH, int NH>
struct ScoreGeom {
  static constexpr int LPP = NCH < 8 ? NCH : 8;       // lanes per position
  static constexpr int CPL = NCH / LPP;               // 16-byte chunks per lane per position (1 or 2)
  static constexpr int PPI = 32 / LPP;                // positions covered by one load instruction
  static constexpr int LD = NH > 1 ? 4 : 8;           // loads per lane per sub-tile (fewer with several heads)
  static constexpr int NP = LD / CPL;                 // position groups per lane per sub-tile
  static constexpr int SUB = NP * PPI;                // positions per sub-tile
  static constexpr int TILE = 2 * SUB;                // positions per warp tile (two sub-tiles)
  static constexpr int OWN = NP / LPP > 0 ? NP / LPP : 1;   // positions a lane owns per sub-tile
};

}  // namespace

size_t select_smem_bytes(const Geometry& g) { return sel_layout(g).total; }

// ===========================================================================
// the kernel
// ===========================================================================
template <int NCH, int NH, bool PG>
__global__ void __launch_bounds__(NT, 1) select_kernel(DecodeParams p) {
  using SG = ScoreGeom<NCH, NH>;
  constexpr int d = NCH * 16;
  const Geometry& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int KR = g.top_k;       // rows attended per request at most (the stride of per-request rows)
  const int BR = g.hot_slots;   // slot rows per (request, layer)
  // page mode: units (what is scored, selected and cached) are pages of PS
  // positions; otherwise PS = 1 and a unit is a position
  constexpr bool paged = PG;
  const int psh = PG ? g.page_shift : 0, PS = 1 << psh;

  extern __shared__ __align__(16) unsigned char smem_raw[];
  const SelLayout L = sel_layout(g);
  __shared__ SelShared sh;
  HS_TRACE(p, 0, 0);

  const bool resolver = (int)blockIdx.x < p.n_resolvers;
  if (resolver) {
    griddep_wait();   // lengths, keys, metadata and scratch of earlier stream work
    griddep_launch_dependents();
  }

  // ======================= scorers =======================
  if (!resolver) {
    int* t_prefix = reinterpret_cast<int*>(smem_raw + L.t_prefix);
    int* t_req = reinterpret_cast<int*>(smem_raw + L.t_req);
    int* t_n = reinterpret_cast<int*>(smem_raw + L.t_n);
    uint32_t* t_thr = reinterpret_cast<uint32_t*>(smem_raw + L.t_thr);
    const int W = (p.sel_grid - p.n_resolvers) * NWARP;
    const int w0 = ((int)blockIdx.x - p.n_resolvers) * NWARP + warp;
    // request of warp tile t, searching forward from request `from`
    auto req_of = [&](int t, int from) {
      int x = from;
      while (t_prefix[x + 1] <= t) ++x;
      return x;
    };
    // the unit rows of warp tile t (request ri) start moving into L2 (one bulk
    // prefetch by lane 0): the register loads of the tile then hit L2, so far more
    // bytes are in flight per SM than the registers hold
    auto prefetch_tile = [&](int t, int ri) {
      const int NU = (t_n[ri] + PS - 1) >> psh;
      const int u0 = (t - t_prefix[ri]) * SG::TILE;
      const int nu = min(SG::TILE, NU - u0);
      if (nu <= 0) return;
      const long long rl = (long long)t_req[ri] * g.n_layers + p.layer;
      if (lane == 0) {
        const int8_t* base =
            paged ? p.s.pbound + rl * (long long)g.max_pages * d : p.s.idx_keys + rl * g.max_context * d;
        bulk_prefetch_l2(base + (long long)u0 * d, (uint32_t)(nu * d));
      } else if (t_thr[ri] != 0u && lane * 32 - 32 < nu) {
        // the tile's page-table entries (read for the candidates it lists), 32 a line
        prefetch_line_l2(p.s.page + rl * g.max_context + u0 + (lane * 32 - 32));
      }
    };
    // warp tiles of every request that needs a selection; returns their number
    auto build_tables = [&]() {
      int carry = 0;
      for (int base = 0; base < p.n_req; base += NT) {
        const int i = base + tid;
        int nt = 0;
        if (i < p.n_req) {
          const int req = p.req_ids ? p.req_ids[i] : i;
          int N = 0;
          uint32_t thr = 0;
          if (req >= 0 && req < g.max_requests) {
            const long long rl = (long long)req * g.n_layers + p.layer;
            N = p.s.length[rl];
            if (p.new_kv && N + 1 <= g.max_context) ++N;   // the token this call appends
            thr = p.s.cand_thr[rl];
          }
          const int NU = (N + PS - 1) >> psh;
          const bool scored = NU > (KR >> psh) && p.role == ROLE_SELECT;
          nt = scored ? (NU + SG::TILE - 1) / SG::TILE : 0;
          t_req[i] = scored ? req : -1;
          t_n[i] = N;
          t_thr[i] = (scored && NH == 1) ? thr : 0u;   // candidate listing: single-head keys only
        }
        int tot;
        const int ex = block_exclusive_scan<NT>(nt, sh.scan, &tot);
        if (i < p.n_req) t_prefix[i] = carry + ex;
        carry += tot;
      }
      if (tid == 0) t_prefix[p.n_req] = carry;
      __syncthreads();
      return carry;
    };

    // lane roles inside a load instruction
    const int pg = lane / SG::LPP;            // position within the instruction
    const int cl = lane % SG::LPP;            // chunk column of the lane
    int4 q[NH][SG::CPL];
    int qw[NH];   // head weights (multi-head indexer)
    int q_r = -1;
    const int qstride = NH > 1 ? NH * d + 16 : g.d_idx;   // bytes of one request's indexer query
    const int hc = g.d_idx / 16;   // page mode: a unit row is [key maxima | key minima], 2 * hc chunks

    // loads of sub-tile `half` of tile t (request ri) into v (zeros past the last
    // unit).  Unit rows: index keys, or in page mode the stored [max | min] bounds
    // of each page; the unit holding this call's appended token combines its key
    // (a page it opens has that key as both bounds).
    auto load_sub = [&](int t, int ri, int half, int4 (&v)[SG::LD]) {
      const int N = t_n[ri];
      const int NU = (N + PS - 1) >> psh;
      const int pos0 = (t - t_prefix[ri]) * SG::TILE + half * SG::SUB;
      const long long rl = (long long)t_req[ri] * g.n_layers + p.layer;
      const int8_t* base = paged ? p.s.pbound + rl * (long long)g.max_pages * d : p.s.idx_keys + rl * g.max_context * d;
      const int newu = p.new_kv ? (N - 1) >> psh : -1;
      const bool fresh = ((N - 1) & (PS - 1)) == 0;   // the appended token opens its page
      const int8_t* nk = p.new_keys + (long long)ri * g.d_idx;
#pragma unroll
      for (int u = 0; u < SG::LD; ++u) {
        const int pos = pos0 + (u / SG::CPL) * SG::PPI + pg;
        const int ch = cl * SG::CPL + (u % SG::CPL);
        v[u] = make_int4(0, 0, 0, 0);
        if (pos < NU) {
          if (pos != newu) {
            v[u] = ld_stream(base + (long long)pos * d + ch * 16);
          } else if (!paged) {
            v[u] = *reinterpret_cast<const int4*>(nk + ch * 16);
          } else {
            const bool hi = ch < hc;
            const int4 kn = *reinterpret_cast<const int4*>(nk + (hi ? ch : ch - hc) * 16);
            if (fresh) {
              v[u] = kn;
            } else {
              const int4 old = ld_stream(base + (long long)pos * d + ch * 16);
              v[u] = hi ? vmax16(old, kn) : vmin16(old, kn);
            }
          }
        }
      }
    };

    // page-table entries of the units this lane owns in tile t (request ri), for
    // the candidates it lists: the resolver then needs no page-table gathers on
    // its critical path.  Read after the grid dependency only (the page table is
    // earlier stream work's), and only for requests that list candidates.
    auto load_pg = [&](int t, int ri, int (&pv)[2][SG::OWN]) {
      const int NU = (t_n[ri] + PS - 1) >> psh;
      const int u0 = (t - t_prefix[ri]) * SG::TILE;
      const int32_t* page_rl = p.s.page + ((long long)t_req[ri] * g.n_layers + p.layer) * g.max_context;
#pragma unroll
      for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int o = 0; o < SG::OWN; ++o) {
          const int pos = u0 + half * SG::SUB + (o * SG::LPP + cl) * SG::PPI + pg;
          pv[half][o] = (t_thr[ri] != 0u && pos < NU) ? __ldcg(page_rl + pos) : -1;
        }
    };

    // Before the grid dependency resolves: the tile map from the state as it
    // stands (the library's own lengths and keys, which no kernel still running
    // writes), this warp's first tile into registers and its second towards L2,
    // overlapping the previous kernel's tail.  The map is rebuilt after the wait;
    // the first tile is loaded again if its place in the map changed, and is
    // loaded only then if it holds this call's appended token (whose key is the
    // caller's input, which may come from the kernel just before).
    int4 va[SG::LD], vb[SG::LD];
    int pre_req = -1, pre_n = -1, pre_off = -1;
    {
      const int total0 = build_tables();
      if (w0 < total0) {
        const int ri0 = req_of(w0, 0);
        pre_n = t_n[ri0];
        pre_off = (w0 - t_prefix[ri0]) * SG::TILE;
        const int newu = p.new_kv ? (pre_n - 1) >> psh : -1;
        if (newu < pre_off || newu >= pre_off + SG::TILE) {
          pre_req = t_req[ri0];
          load_sub(w0, ri0, 0, va);
          load_sub(w0, ri0, 1, vb);
        }
      }
      if (w0 + W < total0) prefetch_tile(w0 + W, req_of(w0 + W, 0));
      __syncthreads();   // the tables are rebuilt below
    }
    griddep_wait();   // lengths, keys, metadata and scratch of earlier stream work
    griddep_launch_dependents();
    const int total = build_tables();
    // this CTA has read every length and threshold it needs
    if (tid == 0) red_release_add(&p.s.sync[0], 1u);
    HS_TRACE(p, 0, 1);
    int r_cur = 0;
    int pgv[2][SG::OWN];   // page-table entries of this lane's units in the current tile
    if (w0 < total) {
      r_cur = req_of(w0, 0);
      const bool same = pre_req >= 0 && t_req[r_cur] == pre_req && t_n[r_cur] == pre_n &&
                        (w0 - t_prefix[r_cur]) * SG::TILE == pre_off;
      if (!same) {
        load_sub(w0, r_cur, 0, va);
        load_sub(w0, r_cur, 1, vb);
      }
      load_pg(w0, r_cur, pgv);
    }
    for (int t = w0; t < total; t += W) {
      const int ri = r_cur;
      const int N = (t_n[ri] + PS - 1) >> psh;   // units of this request
      const int tile0 = (t - t_prefix[ri]) * SG::TILE;
      const uint32_t thr = t_thr[ri];
      if (ri != q_r) {
        q_r = ri;
        const int8_t* qrow = p.q_idx + (long long)ri * qstride;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const int4* qs = reinterpret_cast<const int4*>(qrow + h * d);
#pragma unroll
          for (int c = 0; c < SG::CPL; ++c) {
            const int cc = cl * SG::CPL + c;
            if (!paged) {
              q[h][c] = qs[cc];
            } else {
              // [max(q, 0) | min(q, 0)] against [maxima | minima]: per dimension the
              // larger of q * kmax and q * kmin
              const int4 z = make_int4(0, 0, 0, 0);
              q[h][c] = cc < hc ? vmax16(qs[cc], z) : vmin16(qs[cc - hc], z);
            }
          }
          qw[h] = NH > 1 ? max(0, (int)qrow[NH * d + h]) : 1;   // negative weights count as 0
        }
      }
      uint32_t* keys_out = p.s.scores + (long long)ri * p.score_stride;
      const int tn = t + W;
      const int rn = tn < total ? req_of(tn, ri) : ri;
      // keys of both sub-tiles; lane cl of a position group owns the groups j with
      // j % LPP == cl
      uint32_t ownk[2][SG::OWN];
      int ownp[2][SG::OWN];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int4 (&v)[SG::LD] = half == 0 ? va : vb;
        int acc[SG::NP][NH];   // each head's partial dot product over this lane's chunks
#pragma unroll
        for (int j = 0; j < SG::NP; ++j)
#pragma unroll
          for (int h = 0; h < NH; ++h) acc[j][h] = 0;
#pragma unroll
        for (int u = 0; u < SG::LD; ++u) {
          const int j = u / SG::CPL;
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int4 qq = q[h][u % SG::CPL];
            acc[j][h] = __dp4a(v[u].x, qq.x, acc[j][h]);
            acc[j][h] = __dp4a(v[u].y, qq.y, acc[j][h]);
            acc[j][h] = __dp4a(v[u].z, qq.z, acc[j][h]);
            acc[j][h] = __dp4a(v[u].w, qq.w, acc[j][h]);
          }
        }
        // key of each position group: single head, score + 2^22 (24 bits); several
        // heads, sum_h w_h * max(0, dot_h) (non-negative, below 2^32)
        uint32_t key[SG::NP];
#pragma unroll
        for (int j = 0; j < SG::NP; ++j) {
          unsigned tot = 0;
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            int dh = acc[j][h];
#pragma unroll
            for (int o = 1; o < SG::LPP; o <<= 1) dh += __shfl_xor_sync(FULL_MASK, dh, o);
            if (NH == 1) tot = (unsigned)(dh + IDX_KEY_BIAS);
            else tot += (unsigned)qw[h] * (unsigned)max(dh, 0);
          }
          key[j] = tot;
        }
        const int sub0 = tile0 + half * SG::SUB;
#pragma unroll
        for (int o = 0; o < SG::OWN; ++o) {
          ownk[half][o] = 0;
          ownp[half][o] = N;   // none
        }
#pragma unroll
        for (int j = 0; j < SG::NP; ++j) {
          if (j % SG::LPP == cl) {
            const int o = j / SG::LPP;
            ownp[half][o] = sub0 + j * SG::PPI + pg;
            ownk[half][o] = key[j];
          }
        }
#pragma unroll
        for (int o = 0; o < SG::OWN; ++o)
          if (ownp[half][o] < N) keys_out[ownp[half][o]] = ownk[half][o];
      }
      // the tile's keys at or above the candidate threshold, listed with one atomic
      if (thr != 0u) {
        unsigned mk[2][SG::OWN];
        int cnt = 0;
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int o = 0; o < SG::OWN; ++o) {
            mk[half][o] = __ballot_sync(FULL_MASK, ownp[half][o] < N && ownk[half][o] >= thr);
            cnt += __popc(mk[half][o]);
          }
        if (cnt > 0) {   // warp-uniform
          unsigned base = 0;
          if (lane == 0) base = atomicAdd(p.s.cand_cnt + ri, (unsigned)cnt);
          base = __shfl_sync(FULL_MASK, base, 0);
          const unsigned below = (1u << lane) - 1u;
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int o = 0; o < SG::OWN; ++o) {
              const unsigned at = base + __popc(mk[half][o] & below);
              if (((mk[half][o] >> lane) & 1u) && at < 2u * (unsigned)KR) {
                p.s.cand[(long long)ri * 2 * KR + at] = make_uint2((uint32_t)ownp[half][o], ownk[half][o]);
                p.s.cand_slot[(long long)ri * 2 * KR + at] = pgv[half][o];
              }
              base += __popc(mk[half][o]);
            }
        }
      }
      __syncwarp();
      if (lane == 0) red_release_add(p.s.tiles_done + ri, 1u);
      // then the next tile: its rows two rounds ahead towards L2, and the register
      // loads of the next one (issued after the release, whose fence would
      // otherwise wait for them to land)
      if (tn + W < total) prefetch_tile(tn + W, req_of(tn + W, rn));
      if (tn < total) {
        load_sub(tn, rn, 0, va);
        load_sub(tn, rn, 1, vb);
        load_pg(tn, rn, pgv);
      }
      HS_TRACE_IF(p, 0, 3, tid == 0 && t == w0);
      HS_TRACE_IF(p, 0, 4, tid == 0 && t == w0 + W);
      r_cur = rn;
    }
    HS_TRACE(p, 0, 2);
    return;
  }

  // ======================= resolvers =======================
  // in units: k selected, B slots (page mode: pages and page slots of PS rows)
  const int K = KR >> psh, B = BR >> psh;
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
  static_assert(IDX_BINS % (4 * NT) == 0, "whole 16-byte histogram chunks per thread");

  for (int ri = (int)blockIdx.x; ri < p.n_req; ri += p.n_resolvers) {
    HS_TRACE_IF(p, 1, 0, tid == 0 && ri == (int)blockIdx.x);
    int32_t* sel_out = p.sel_out ? p.sel_out + (long long)ri * KR : nullptr;
    const int req = p.req_ids ? p.req_ids[ri] : ri;
    if (req < 0 || req >= g.max_requests) {
      if (tid == 0) set_error(p.s.dev_error, HS_DEVERR_REQ_RANGE);
      if (sel_out)
        for (int i = tid; i < KR; i += NT) sel_out[i] = -1;
      if (p.publish) {
        __syncthreads();
        if (tid == 0) {
          __threadfence();
          st_release(p.s.ready + ri, 1u);   // k_eff + 1 = 1: nothing selected
        }
      }
      __syncthreads();
      continue;
    }
    const long long rl = (long long)req * g.n_layers + p.layer;
    for (int j = tid; j < B; j += NT) used[j] = 0;

    // ---- 0. every read that does not depend on the scores, issued together ----
    const int32_t* order_g = p.s.order + rl * BR;
    for (int c4 = tid; c4 < B / 4; c4 += NT) cp_async_16(ord + 4 * c4, order_g + 4 * c4);
    if (L.rev_smem) {
      const int32_t* rev_g = p.s.reverse + rl * BR;
      for (int c4 = tid; c4 < B / 4; c4 += NT) cp_async_16(rev_s + 4 * c4, rev_g + 4 * c4);
    }
    if (p.new_kv) {
      for (int v = tid; v < g.row_bytes / 16; v += NT)
        cp_async_16(newrow + 16 * v,
                    reinterpret_cast<const unsigned char*>(p.new_kv + (long long)ri * g.row_elems) + 16 * v);
      if (tid < g.d_idx / 16) cp_async_16(newkey + 16 * tid, p.new_keys + (long long)ri * g.d_idx + 16 * tid);
    }
    if (tid == 0) {
      const int len = p.s.length[rl];
      sh.len = len;
      sh.t_step = p.s.step[rl];
      sh.thr = p.s.cand_thr[rl];
      int N = len;
      if (p.new_kv) {
        if (len + 1 <= g.max_context) N = len + 1;
        else set_error(p.s.dev_error, HS_DEVERR_CAPACITY);
      }
      sh.N = N;
      sh.ok = 1;
      const int NUt = (N + PS - 1) >> psh;
      if (N == 0) set_error(p.s.dev_error, HS_DEVERR_EMPTY);   // nothing to attend: the output is 0
      if (p.role == ROLE_GIVEN) {   // the lead of this step must have left a selection of this length
        const bool armed = p.s.sh_armed[rl] != 0 && p.s.sh_kk[rl] == min(K, NUt);
        p.s.sh_armed[rl] = 0;
        if (!armed) {
          set_error(p.s.dev_error, HS_DEVERR_NO_LEAD);
          sh.ok = 0;
        }
      }
      sh.thr_next = 0u;
      if (NUt > K && p.role == ROLE_SELECT) {   // wait until every tile of this request is scored
        const unsigned ntile = (unsigned)((NUt + SG::TILE - 1) / SG::TILE);
        if (!wait_counter(p.s.tiles_done + ri, ntile)) {
          set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
          sh.ok = 0;
        }
        p.s.tiles_done[ri] = 0;   // ready for the next call
      }
      sh.cnt = 0;
    }
    cp_async_wait_all();
    __syncthreads();
    HS_TRACE_IF(p, 1, 1, tid == 0 && ri == (int)blockIdx.x);
    const int len = sh.len, Np = sh.N, t_step = sh.t_step;   // Np positions with the appended token
    const int N = (Np + PS - 1) >> psh;                        // units
    const bool appended = Np > len;
    const int kk = sh.ok ? min(K, N) : 0;   // (a given selection has the same k_eff: same N)
    // the candidate list (every entry it can hold: those past the count are
    // ignored) and its count, in one round trip
    uint2 cv[CAND_REG];
    if (N > K && p.role == ROLE_SELECT) {   // CTA-uniform
      const bool may_cand = sh.ok && L.fast && N <= FAST_MAX_N && sh.thr != 0u;
      const uint2* cl = p.s.cand + (long long)ri * 2 * KR;
      const int cap = min(2 * KR, CAND_REG * NT);
#pragma unroll
      for (int j = 0; j < CAND_REG; ++j) {
        const int i = tid + j * NT;
        cv[j] = (may_cand && i < cap) ? __ldcg(cl + i) : make_uint2(0u, 0u);
      }
      if (tid == 0) {
        sh.cnt = (int)min(__ldcg(p.s.cand_cnt + ri), 0x7fffffffu);
        p.s.cand_cnt[ri] = 0;
      }
      __syncthreads();
    }

    // ======================= 1. top-k, ascending =======================
    // The previous call's threshold listed between k and min(2k, 4096) keys: the k
    // largest (ties included) are all in the list, held in registers here.
    const bool use_cand = sh.ok && N > K && L.fast && N <= FAST_MAX_N && sh.thr != 0u &&
                          sh.cnt >= K && sh.cnt <= min(2 * K, CAND_REG * NT);
    bool slots_known = false;   // the candidate path reads each selected position's page entry itself
    // the candidate path (rows, not pages) also writes the selection, marks the
    // hits used and writes their slots as it emits them: no later passes for those
    bool emitted_out = false, bad_pre = false;
    // the next call lists keys at or above the exact key of rank 1.5 k (found after
    // publication): about 1.5 k of them, half way between k and the list's room
    const int k_next = (int)min((long long)N, (long long)K + K / 2);
    if (tid == 0) sh.thr_src = 0;
    if (!sh.ok) {
      // scores incomplete: nothing selected (the output of this request is 0)
    } else if (p.role == ROLE_GIVEN) {
      // the selection this layer's group lead left for it (same step, same positions)
      const int32_t* gsel = p.s.sh_sel + rl * KR;
      for (int i = tid; i < kk; i += NT) sel[i] = __ldcg(gsel + i);
    } else if (N <= K) {
      for (int i = tid; i < N; i += NT) sel[i] = i;
    } else if (use_cand) {
      const int cnt = sh.cnt;
      const int NWd = (N + 31) >> 5;
      uint32_t* gtw = bitmap;                         // [NWd] positions whose key is above the k-th
      uint32_t* tiw = bitmap + FAST_MAX_N / 32;       // [NWd] positions whose key equals it
      uint16_t* gpre = reinterpret_cast<uint16_t*>(smem_raw + L.wpre);   // [NWd] above-threshold positions before each word
      uint16_t* epre = gpre + FAST_MAX_N / 32;                           // [NWd] ties before each word (all < 2^16)
      int cpg[CAND_REG];
      // every selected position is a candidate: its page entry, listed with it by
      // the scorer, is the hit test
      const int32_t* csl = p.s.cand_slot + (long long)ri * 2 * KR;
#pragma unroll
      for (int j = 0; j < CAND_REG; ++j) cpg[j] = tid + j * NT < cnt ? __ldcg(csl + tid + j * NT) : -1;
      for (int c = tid; c < IDX_BINS / 4; c += NT) reinterpret_cast<uint4*>(h)[c] = make_uint4(0, 0, 0, 0);
      for (int w = tid; w < NWd; w += NT) {
        gtw[w] = 0u;
        tiw[w] = 0u;
      }
      __syncthreads();
      HS_TRACE_IF(p, 1, 10, tid == 0 && ri == (int)blockIdx.x);
#pragma unroll
      for (int j = 0; j < CAND_REG; ++j)
        if (tid + j * NT < cnt) atomicAdd(&h[cv[j].y >> 12], 1u);
      __syncthreads();
      HS_TRACE_IF(p, 1, 11, tid == 0 && ri == (int)blockIdx.x);
      select_digit(h, K, sh.scan, &sh.b1, &sh.above1, cnt >= k_next ? k_next : 0, &sh.bt, &sh.above_t);
      if (cnt >= k_next) {
        if (tid == 0) {
          sh.thr_next = (uint32_t)sh.bt << 12;
          sh.thr_src = 1;
        }
      } else if (tid == 0) {
        sh.thr_next = sh.thr;   // the list held fewer: keep the threshold that gave >= k
      }
      if (tid == 0 && N > CAND_MAX_N_PER_K * K) sh.thr_next = 0u;
      const int b1 = sh.b1, above1 = sh.above1;
      for (int c = tid; c < IDX_BINS / 4; c += NT) reinterpret_cast<uint4*>(h)[c] = make_uint4(0, 0, 0, 0);
      __syncthreads();
#pragma unroll
      for (int j = 0; j < CAND_REG; ++j)
        if (tid + j * NT < cnt && (int)(cv[j].y >> 12) == b1) atomicAdd(&h[cv[j].y & 4095u], 1u);
      __syncthreads();
      HS_TRACE_IF(p, 1, 2, tid == 0 && ri == (int)blockIdx.x);
      select_digit(h, K - above1, sh.scan, &sh.b2, &sh.above2);
      const uint32_t vstar = ((uint32_t)b1 << 12) | (uint32_t)sh.b2;
      const int need_eq = K - (above1 + sh.above2);   // >= 1
#pragma unroll
      for (int j = 0; j < CAND_REG; ++j)
        if (tid + j * NT < cnt) {
          const uint32_t pp = cv[j].x;
          if (cv[j].y > vstar) atomicOr(&gtw[pp >> 5], 1u << (pp & 31));
          else if (cv[j].y == vstar) atomicOr(&tiw[pp >> 5], 1u << (pp & 31));
        }
      __syncthreads();
      // per-word prefix counts of the taken-above and tie positions (each thread a
      // contiguous range of words)
      const int WPT = (NWd + NT - 1) / NT;
      const int w0 = min(NWd, tid * WPT), w1 = min(NWd, w0 + WPT);
      int ng = 0, ne = 0;
      for (int w = w0; w < w1; ++w) {
        ng += __popc(gtw[w]);
        ne += __popc(tiw[w]);
      }
      const int2 ex = block_exclusive_scan2<NT>(ng, ne, sh.scan, nullptr, nullptr);
      int rg = ex.x, re = ex.y;
      for (int w = w0; w < w1; ++w) {
        gpre[w] = (uint16_t)rg;
        epre[w] = (uint16_t)re;
        rg += __popc(gtw[w]);
        re += __popc(tiw[w]);
      }
      __syncthreads();
      HS_TRACE_IF(p, 1, 3, tid == 0 && ri == (int)blockIdx.x);
      // each taken candidate's place in the ascending output: the taken positions
      // before it (all above-threshold ones, ties only up to need_eq)
#pragma unroll
      for (int j = 0; j < CAND_REG; ++j)
        if (tid + j * NT < cnt) {
          const uint32_t pp = cv[j].x;
          const int w = (int)(pp >> 5);
          const uint32_t lm = (1u << (pp & 31)) - 1u;
          const int gb = gpre[w] + __popc(gtw[w] & lm);
          const int eb = epre[w] + __popc(tiw[w] & lm);
          const bool taken = cv[j].y > vstar || (cv[j].y == vstar && eb < need_eq);
          if (taken) {
            const int idx = gb + min(eb, need_eq);
            sel[idx] = (int)pp;
            slot_sel[idx] = cpg[j];
            if (!paged) {
              p.s.sel[(long long)ri * KR + idx] = (int)pp;
              const int s4 = cpg[j];
              if (s4 >= B) {
                bad_pre = true;
              } else if (s4 >= 0) {
                used[s4] = 1;
                p.s.slot_of_sel[(long long)ri * KR + idx] = s4;
              }
            }
          }
        }
      slots_known = true;
      emitted_out = !paged;
    } else if (NH > 1) {
      // the multi-head indexer's 32-bit keys: three digits (12, 12 and 8 bits),
      // each found by a histogram pass over the keys of the digits above it, then
      // a counting pass and the ascending emission (ties to the lower position)
      const uint32_t* keys = p.s.scores + (long long)ri * p.score_stride;
      const uint4* k4 = reinterpret_cast<const uint4*>(keys);   // rows padded to a multiple of 4 keys
      const int n4 = N >> 2;
      int above = 0;
      uint32_t prefix = 0;   // the digits found so far
      constexpr int SHIFT[3] = {20, 8, 0};
      constexpr uint32_t MASK[3] = {4095u, 4095u, 255u};
#pragma unroll 1
      for (int dgt = 0; dgt < 3; ++dgt) {
        for (int c = tid; c < IDX_BINS / 4; c += NT) reinterpret_cast<uint4*>(h)[c] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        const int sh_d = SHIFT[dgt];
        const int sh_p = dgt == 0 ? 32 : SHIFT[dgt - 1];   // keys whose higher digits match `prefix`
        auto count = [&](uint32_t k) {
          if (sh_p == 32 || (k >> sh_p) == prefix) atomicAdd(&h[(k >> sh_d) & MASK[dgt]], 1u);
        };
        constexpr int UA = 8;
        for (int i0 = tid; i0 < n4; i0 += UA * NT) {
          uint4 v[UA];
#pragma unroll
          for (int u = 0; u < UA; ++u) {
            const int i = i0 + u * NT;
            v[u] = i < n4 ? __ldcg(k4 + i) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < UA; ++u)
            if (i0 + u * NT < n4) {
              count(v[u].x);
              count(v[u].y);
              count(v[u].z);
              count(v[u].w);
            }
        }
        for (int i = 4 * n4 + tid; i < N; i += NT) count(__ldcg(keys + i));
        __syncthreads();
        select_digit(h, K - above, sh.scan, &sh.b1, &sh.above1);
        above += sh.above1;
        prefix = (prefix << (dgt == 0 ? 0 : (SHIFT[dgt - 1] - SHIFT[dgt]))) | (uint32_t)sh.b1;
        __syncthreads();
      }
      const uint32_t vstar = prefix;   // the k-th largest key
      const int need_eq = K - above;   // >= 1
      if (tid == 0) sh.thr_next = 0u;  // no candidate listing for these keys
      const int per = ((N + NT - 1) / NT + 3) & ~3;
      const int j0 = min(N, tid * per), j1 = min(N, j0 + per);
      int n_gt = 0, n_eq = 0;
      for (int j = j0; j < j1; j += 4) {   // multiples of 4 in bounds (padded rows)
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(keys + j));
        const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (j + e < j1) {
            n_gt += kv[e] > vstar;
            n_eq += kv[e] == vstar;
          }
      }
      const int2 before = block_exclusive_scan2<NT>(n_gt, n_eq, sh.scan, nullptr, nullptr);
      int o = before.x + min(before.y, need_eq);
      int eq_rank = before.y;
      for (int j = j0; j < j1; j += 4) {
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(keys + j));
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
    } else {
      const uint32_t* keys = p.s.scores + (long long)ri * p.score_stride;
      const bool fast = L.fast && N <= FAST_MAX_N;
      if (tid == 0) red_add_u64(&p.s.glob[2], 1ull);   // a selection over every key
      for (int c = tid; c < IDX_BINS / 4; c += NT) reinterpret_cast<uint4*>(h)[c] = make_uint4(0, 0, 0, 0);
      __syncthreads();
      // first-digit histogram: when the candidate list only overflowed, every one of
      // the k largest keys clears the threshold, so only those keys are counted;
      // else all keys
      {
        const uint32_t floor_key = (sh.thr != 0u && sh.cnt >= K) ? sh.thr : 0u;
        const uint4* k4 = reinterpret_cast<const uint4*>(keys);   // rows padded to a multiple of 4 keys
        const int n4 = N >> 2;
        auto hadd = [&](uint32_t k) {
          if (k >= floor_key) atomicAdd(&h[k >> 12], 1u);
        };
        constexpr int UA = 8;
        for (int i0 = tid; i0 < n4; i0 += UA * NT) {
          uint4 v[UA];
#pragma unroll
          for (int u = 0; u < UA; ++u) {
            const int i = i0 + u * NT;
            v[u] = i < n4 ? __ldcg(k4 + i) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < UA; ++u)
            if (i0 + u * NT < n4) {
              hadd(v[u].x);
              hadd(v[u].y);
              hadd(v[u].z);
              hadd(v[u].w);
            }
        }
        for (int i = 4 * n4 + tid; i < N; i += NT) {
          const uint32_t k = __ldcg(keys + i);
          if (k >= floor_key) atomicAdd(&h[k >> 12], 1u);
        }
      }
      __syncthreads();
      // the digit of the k-th largest key, and the digit above which ~1.25 k keys
      // lie: the next call lists keys from there on (exact whenever >= k clear it)
      const int counted = (sh.thr != 0u && sh.cnt >= K) ? sh.cnt : N;   // keys the histogram holds
      select_digit(h, K, sh.scan, &sh.b1, &sh.above1, counted >= k_next ? k_next : 0, &sh.bt, &sh.above_t);
      if (counted >= k_next) {
        if (tid == 0) {
          sh.thr_next = (uint32_t)sh.bt << 12;
          sh.thr_src = 2;
        }
      } else if (tid == 0) {
        sh.thr_next = sh.thr;
      }
      const int b1 = sh.b1, above1 = sh.above1;
      // listing costs the scorers about as much per position as the full pass
      // costs here, so it pays only while the context is short relative to k
      if (tid == 0 && N > CAND_MAX_N_PER_K * K) sh.thr_next = 0u;
      for (int c = tid; c < IDX_BINS / 4; c += NT) reinterpret_cast<uint4*>(h)[c] = make_uint4(0, 0, 0, 0);
      __syncthreads();
      // per-thread contiguous ranges (the rescan path)
      const int per = ((N + NT - 1) / NT + 3) & ~3;
      const int j0 = min(N, tid * per), j1 = min(N, j0 + per);
      // per-warp contiguous chunks of 128 positions (the one-pass path)
      const int wid = warp;
      const int NC = (N + 127) >> 7;
      const int c0 = (int)((long long)wid * NC / NWARP), c1 = (int)((long long)(wid + 1) * NC / NWARP);
      uint32_t* wl = lists + wid * WCAP;
      int wcnt = 0;       // entries of this warp's list (warp-uniform)
      int lane_gt = 0;    // keys above digit b1 seen by this lane
      bool overflow = false;
      if (fast) {
        const uint4* k4 = reinterpret_cast<const uint4*>(keys);
        constexpr int UC = 8;   // chunks in flight per lane
        for (int cb = c0; cb < c1; cb += UC) {
          uint4 v[UC];
#pragma unroll
          for (int u = 0; u < UC; ++u) {
            const int pos = 128 * (cb + u) + 4 * lane;
            v[u] = (cb + u < c1 && pos < N) ? __ldcg(k4 + (cb + u) * 32 + lane) : make_uint4(0, 0, 0, 0);
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
        constexpr int UA = 8;
        for (int i0 = tid; i0 < n4; i0 += UA * NT) {
          uint4 v[UA];
#pragma unroll
          for (int u = 0; u < UA; ++u) {
            const int i = i0 + u * NT;
            v[u] = i < n4 ? __ldcg(k4 + i) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < UA; ++u) {
            if ((int)(v[u].x >> 12) == b1) atomicAdd(&h[v[u].x & 4095u], 1u);
            if ((int)(v[u].y >> 12) == b1) atomicAdd(&h[v[u].y & 4095u], 1u);
            if ((int)(v[u].z >> 12) == b1) atomicAdd(&h[v[u].z & 4095u], 1u);
            if ((int)(v[u].w >> 12) == b1) atomicAdd(&h[v[u].w & 4095u], 1u);
          }
        }
        for (int i = 4 * n4 + tid; i < N; i += NT) {
          const uint32_t v = __ldcg(keys + i);
          if ((int)(v >> 12) == b1) atomicAdd(&h[v & 4095u], 1u);
        }
      }
      // the barrier is taken on every path (it orders the histogram atomics above
      // before the digit select below), then decides whether the lists are usable
      const bool any_overflow = __syncthreads_or(overflow);
      const bool use_lists = fast && !any_overflow;
      select_digit(h, K - above1, sh.scan, &sh.b2, &sh.above2);
      const int b2 = sh.b2;
      const uint32_t vstar = ((uint32_t)b1 << 12) | (uint32_t)b2;
      const int need_eq = K - (above1 + sh.above2);   // >= 1
      if (use_lists) {
        int n_gt = lane_gt, n_eq = 0;
        for (int qq = lane; qq < wcnt; qq += 32) {
          const int lo = (int)(wl[qq] & 4095u);
          n_gt += lo > b2;
          n_eq += lo == b2;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          n_gt += __shfl_xor_sync(FULL_MASK, n_gt, o);
          n_eq += __shfl_xor_sync(FULL_MASK, n_eq, o);
        }
        const int2 wb =
            block_exclusive_scan2<NT>(lane == 0 ? n_gt : 0, lane == 0 ? n_eq : 0, sh.scan, nullptr, nullptr);
        const int gt_before = __shfl_sync(FULL_MASK, wb.x, 0), eq_before = __shfl_sync(FULL_MASK, wb.y, 0);
        // emission: lane l owns bitmap word q0 + l of each group of 32 words
        int out = gt_before + min(eq_before, need_eq);
        int tie_run = eq_before;   // ties before the current list entry (position order)
        int qe = 0;                // next list entry
        const int w_end = 4 * c1;
        for (int q0 = 4 * c0; q0 < w_end; q0 += 32) {
          const int qq = q0 + lane;
          uint32_t m = qq < w_end ? bitmap[qq] : 0u;
          for (; qe < wcnt; ++qe) {   // list entries of this group of words, in order
            const uint32_t e = wl[qe];
            const int pos = (int)(e >> 12);
            if ((pos >> 5) >= q0 + 32) break;
            const int lo = (int)(e & 4095u);
            const bool mine = (pos >> 5) == qq;
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
            if (o < K) sel[o++] = 32 * qq + bb;
          }
          out += __shfl_sync(FULL_MASK, incl, 31);
        }
      } else {
        int n_gt = 0, n_eq = 0;
        for (int j = j0; j < j1; j += 4) {   // multiples of 4 in bounds (padded rows)
          const uint4 v = __ldcg(reinterpret_cast<const uint4*>(keys + j));
          const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (j + e < j1) {
              n_gt += kv[e] > vstar;
              n_eq += kv[e] == vstar;
            }
        }
        const int2 before = block_exclusive_scan2<NT>(n_gt, n_eq, sh.scan, nullptr, nullptr);
        int o = before.x + min(before.y, need_eq);
        int eq_rank = before.y;
        for (int j = j0; j < j1; j += 4) {
          const uint4 v = __ldcg(reinterpret_cast<const uint4*>(keys + j));
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
    HS_TRACE_IF(p, 1, 4, tid == 0 && ri == (int)blockIdx.x);
    // rows attended: every position of the selected units below the length (only
    // the last page can be partial; when selected it is the last selected unit)
    const int kkr = !paged ? kk : (kk > 0 ? kk * PS - (sel[kk - 1] == N - 1 ? N * PS - Np : 0) : 0);
    // the selection for the attention kernel now; the caller's copy (sel_out)
    // after publication
    auto row_pos = [&](int i) { return paged ? (sel[i >> psh] << psh) + (i & (PS - 1)) : sel[i]; };
    int32_t* sel_g = p.s.sel + (long long)ri * KR;
    if (!emitted_out)
      for (int i = tid; i < kkr; i += NT) sel_g[i] = row_pos(i);

    // ======================= 2. RESOLVE metadata =======================
    // pass 0: this call's layer.  Passes 1..n_follow: the follower layers of its
    // group, which share this selection: each is resolved against its own page
    // table and LRU list now, and its missed rows are pulled into its slots ahead
    // of its own call (all but its appended token, whose row comes with that call).
    bool skip_rest = false;
    const int n_pass = 1 + ((p.role == ROLE_SELECT && p.share_prefetch && sh.ok) ? p.n_follow : 0);
    for (int pass = 0; pass < n_pass; ++pass) {
    const long long rlx = rl + pass;
    if (pass > 0) {
      __syncthreads();   // the previous pass is done with the shared arrays
      for (int j = tid; j < B; j += NT) used[j] = 0;
      const int32_t* order_f = p.s.order + rlx * BR;
      for (int c4 = tid; c4 < B / 4; c4 += NT) cp_async_16(ord + 4 * c4, order_f + 4 * c4);
      if (L.rev_smem) {
        const int32_t* rev_f = p.s.reverse + rlx * BR;
        for (int c4 = tid; c4 < B / 4; c4 += NT) cp_async_16(rev_s + 4 * c4, rev_f + 4 * c4);
      }
      if (tid == 0) {
        sh.t_step_f = p.s.step[rlx];
        sh.len_f = p.s.length[rlx];
        if (sh.len_f != len) set_error(p.s.dev_error, HS_DEVERR_METADATA);   // layers must move in step
      }
      cp_async_wait_all();
      __syncthreads();
      if (sh.len_f != len) continue;
    }
    int32_t* page = p.s.page + rlx * g.max_context;
    int32_t* reverse = p.s.reverse + rlx * BR;
    int32_t* stamp = p.s.stamp + rlx * BR;
    int32_t* order = p.s.order + rlx * BR;
    int32_t* sos = p.s.slot_of_sel + (long long)ri * KR;
    const int t = pass == 0 ? t_step : sh.t_step_f;
    int m = 0;
    // the lead copies its missed rows in fetch mode 1 (else the attention kernel
    // does); a follower layer always gets its rows now: that is the prefetch
    const bool pull = pass > 0 || p.fetch_mode == 1;
    bool bad = false;
    if (kk > 0 && slots_known && pass == 0) {
      bad = bad_pre;
      if (!emitted_out)
        for (int i = tid; i < kk; i += NT) {
          const int s4 = slot_sel[i];
          if (s4 >= B) bad = true;
          if (s4 >= 0 && s4 < B) used[s4] = 1;
        }
    } else if (kk > 0) {
      // hit test: independent page-table gathers, four in flight per thread
      for (int i0 = tid; i0 < kk; i0 += 4 * NT) {
        int pos[4], s4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * NT;
          pos[u] = i < kk ? sel[i] : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) s4[u] = (pos[u] >= 0 && pos[u] < N) ? page[pos[u]] : -1;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * NT;
          if (i < kk) {
            if (pos[u] < 0 || pos[u] >= N || s4[u] >= B) bad = true;
            slot_sel[i] = s4[u];
            if (s4[u] >= 0 && s4[u] < B) {
              used[s4[u]] = 1;
              if (pass == 0 && !paged) sos[i] = s4[u];   // a hit's slot (misses get theirs below)
            }
          }
        }
      }
    }
    // write-allocate: the token this call appends counts as used even when the
    // selection does not take it (one extra entry after the selection: a new
    // position, so never resident)
    const int extra = (p.write_allocate && !paged && appended && sh.ok && !(kk > 0 && sel[kk - 1] == len)) ? 1 : 0;
    const int kx = kk + extra;
    if (extra && tid == 0) {
      sel[kk] = len;
      slot_sel[kk] = -1;
    }
    if (__syncthreads_or(bad)) {
      // inconsistent metadata: publish nothing usable for this request
      if (tid == 0) set_error(p.s.dev_error, HS_DEVERR_METADATA);
      if (pass == 0 && p.publish && tid == 0) {
        __threadfence();
        st_release(p.s.ready + ri, 1u);   // k_eff + 1 = 1: nothing selected
      }
      skip_rest = pass == 0;
      __syncthreads();
      break;
    }
    HS_TRACE_IF(p, 1, 5, tid == 0 && pass == 0 && ri == (int)blockIdx.x);
    // misses in ascending selection order, and the unpinned entries of the LRU
    // list: warp w takes the w-th contiguous segment of each, counts it by ballots
    // (lane-strided: no shared-memory bank conflicts), one block scan places the
    // segments, and each warp emits its own in order
    const unsigned lt = (1u << lane) - 1u;
    const int segi = (kx + NT - 1) / NT * 32, segj = (B + NT - 1) / NT * 32;
    const int wi0 = min(kx, warp * segi), wi1 = min(kx, wi0 + segi);
    const int wj0 = min(B, warp * segj), wj1 = min(B, wj0 + segj);
    const bool lru_list = p.replacement != HS_REPLACE_RANDOM;
    int nm = 0, nc = 0;
#pragma unroll 4
    for (int i = wi0; i < wi1; i += 32) nm += __popc(__ballot_sync(FULL_MASK, i + lane < wi1 && slot_sel[i + lane] < 0));
    if (lru_list) {
#pragma unroll 4
      for (int j = wj0; j < wj1; j += 32)
        nc += __popc(__ballot_sync(FULL_MASK, j + lane < wj1 && used[ord[j + lane]] == 0));
    }
    const int2 mc = block_exclusive_scan2<NT>(lane == 0 ? nm : 0, lane == 0 ? nc : 0, sh.scan, &m, nullptr);
    int mb = __shfl_sync(FULL_MASK, mc.x, 0);
    // the misses the attention kernel will fetch go to its prefetcher at once
    const bool list_misses = pass == 0 && !pull && p.publish;
    int32_t* mpos = p.s.miss_pos + (long long)ri * KR;
    for (int i = wi0; i < wi1; i += 32) {
      const int ii = i + lane;
      const bool miss = ii < wi1 && slot_sel[ii] < 0;
      const unsigned bal = __ballot_sync(FULL_MASK, miss);
      if (miss) {
        const int at = mb + __popc(bal & lt);
        if (list_misses && ii < kk) mpos[at] = (!paged && appended && sel[ii] == len) ? -1 : sel[ii];
        miss_i[at] = ii;
      }
      mb += __popc(bal);
    }
    if (p.replacement == HS_REPLACE_RANDOM) {
      // victims: the m unpinned slots ranked first (never-filled, then smallest
      // (key, slot)), in ascending slot order.  Two 12-bit digit selections over
      // the 24-bit ranks, then each thread takes its ranks above the threshold
      // and, in slot order, the threshold ties still needed.  "Never filled" is
      // read from the reverse map as it was before this call.
      if (m > 0) {
        const int per_j = (B + NT - 1) / NT;   // a contiguous range of slots per thread
        const int j0 = min(B, tid * per_j), j1 = min(B, j0 + per_j);
        const unsigned long long seed = p.replacement_seed;
        auto rank_of = [&](int j) {
          const int old = L.rev_smem ? rev_s[j] : reverse[j];
          return random_ikey(seed, rlx, t, j, old < 0);
        };
        for (int c = tid; c < IDX_BINS / 4; c += NT) reinterpret_cast<uint4*>(h)[c] = make_uint4(0, 0, 0, 0);
        __syncthreads();
        for (int j = j0; j < j1; ++j)
          if (used[j] == 0) atomicAdd(&h[rank_of(j) >> 12], 1u);
        __syncthreads();
        select_digit(h, m, sh.scan, &sh.rb1, &sh.rabove1);
        const int rb1 = sh.rb1, rab1 = sh.rabove1;
        for (int c = tid; c < IDX_BINS / 4; c += NT) reinterpret_cast<uint4*>(h)[c] = make_uint4(0, 0, 0, 0);
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
        const int2 ex = block_exclusive_scan2<NT>(n_gt, n_eq, sh.scan, nullptr, nullptr);
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
      int cb = __shfl_sync(FULL_MASK, mc.y, 0);
      for (int j = wj0; j < wj1 && cb < m; j += 32) {   // warp-uniform
        const int jj = j + lane;
        const int sl = jj < wj1 ? ord[jj] : 0;
        const bool fr = jj < wj1 && used[sl] == 0;
        const unsigned bal = __ballot_sync(FULL_MASK, fr);
        if (fr) {
          const int at = cb + __popc(bal & lt);
          if (at < m) {
            victim[at] = sl;
            used[sl] = 2;
          }
        }
        cb += __popc(bal);
      }
    }
    __syncthreads();
    if (list_misses && tid == 0) p.s.miss_cnt[ri] = (unsigned)(m - extra) + 1u;   // a hint: no ordering
    HS_TRACE_IF(p, 1, 6, tid == 0 && pass == 0 && ri == (int)blockIdx.x);
    // evict, then record the new residents (stores only); slot of every selected
    // row, misses flagged when the attention kernel copies them
    for (int qq = tid; qq < m; qq += NT) {
      const int v = victim[qq];
      const int i = miss_i[qq];
      const int pnew = sel[i];
      const int old = L.rev_smem ? rev_s[v] : reverse[v];
      if (old >= 0 && old < g.max_context) page[old] = -1;
      reverse[v] = pnew;
      page[pnew] = v;
      slot_sel[i] = v;
      // the lead's appended token: its row is in shared memory, it goes to its slot
      // here; a follower's appended token: flagged, its row comes with its own call.
      // Page mode: a page is flagged whole; its appended row is left out below.
      if (pass == 0) miss_i[qq] = (pull || (!paged && appended && pnew == len)) ? i : (i | HS_SLOT_MISS_FLAG);
      else miss_i[qq] = (appended && pnew == len) ? (i | HS_SLOT_MISS_FLAG) : i;
      // a missed row's slot, flagged when the attention kernel copies it (the
      // hits' slots were written with the hit test)
      if (pass == 0 && !paged && i < kk) sos[i] = (miss_i[qq] & HS_SLOT_MISS_FLAG) ? (v | HS_SLOT_MISS_FLAG) : v;
    }
    __syncthreads();
    if (pass == 0 && !paged) {
      // every selected row's slot is written
    } else if (pass == 0) {
      // page mode: row i of the expansion is row i % PS of page slot slot_sel[i / PS]
      for (int i = tid; i < kkr; i += NT) sos[i] = (slot_sel[i >> psh] << psh) + (i & (PS - 1));
      __syncthreads();
      for (int e = tid; e < m * PS; e += NT) {
        const int qq = e >> psh, o = e & (PS - 1);
        if (!(miss_i[qq] & HS_SLOT_MISS_FLAG)) continue;
        const int u = miss_i[qq] & ~HS_SLOT_MISS_FLAG;
        const int i = (u << psh) + o;
        if (i < kkr && !(appended && (sel[u] << psh) + o == len)) sos[i] |= HS_SLOT_MISS_FLAG;
      }
    } else {   // what the follower's own call needs: selection, slots, k_eff, the pending slot
      int32_t* fs = p.s.sh_slots + rlx * KR;
      int32_t* fp = p.s.sh_sel + rlx * KR;
      for (int i = tid; i < kk; i += NT) {
        fs[i] = slot_sel[i];
        fp[i] = sel[i];
      }
      if (tid == 0) {
        int pend = -1;
        if (m > 0 && (miss_i[m - 1] & HS_SLOT_MISS_FLAG)) pend = victim[m - 1];
        p.s.sh_pend[rlx] = pend;
        p.s.sh_kk[rlx] = kk;
      }
    }

    // ======================= 3. rows this kernel copies into their slots =======================
    // fetch mode 1: every missed row from the host copy; otherwise only the
    // appended token's (from its input copy)
    {
      const int rvec = g.row_bytes / 16;
      const unsigned char* src_base =
          reinterpret_cast<const unsigned char*>(p.s.host_kv) + (size_t)rlx * g.max_context * g.row_bytes;
      unsigned char* dst_base = reinterpret_cast<unsigned char*>(p.s.hot) + (size_t)rlx * BR * g.row_bytes;
      bool wrote = false;   // this call wrote slot rows (CTA-uniform)
      if (paged) {
        // every row of a missed page below the length (fetch mode 1), then the
        // appended row into its page's slot whenever that page is resident: a hit,
        // a page filled by this call, or a resident page the selection passed over
        if (pull) {
          wrote = m > 0;
          const long long total = (long long)m * PS * rvec;
          constexpr int U = 8;
          for (long long e0 = tid; e0 < total; e0 += (long long)U * NT) {
            int4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const long long e = e0 + (long long)u * NT;
              if (e < total) {
                const int qo = (int)(e / rvec);
                const int cidx = (int)(e - (long long)qo * rvec);
                const int pos = (sel[miss_i[qo >> psh]] << psh) + (qo & (PS - 1));
                if (pos >= Np) continue;
                v[u] = (appended && pos == len)
                           ? reinterpret_cast<const int4*>(newrow)[cidx]
                           : *reinterpret_cast<const int4*>(src_base + (size_t)pos * g.row_bytes + cidx * 16);
              }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const long long e = e0 + (long long)u * NT;
              if (e < total) {
                const int qo = (int)(e / rvec);
                const int cidx = (int)(e - (long long)qo * rvec);
                const int o = qo & (PS - 1);
                if ((sel[miss_i[qo >> psh]] << psh) + o >= Np) continue;
                *reinterpret_cast<int4*>(dst_base + (size_t)((victim[qo >> psh] << psh) + o) * g.row_bytes +
                                         cidx * 16) = v[u];
              }
            }
          }
        }
        if (appended) {
          const int ps = page[len >> psh];
          if (ps >= 0 && ps < B) wrote = true;
          if (ps >= 0 && ps < B)
            for (int v = tid; v < rvec; v += NT)
              *reinterpret_cast<int4*>(dst_base + (size_t)((ps << psh) + (len & (PS - 1))) * g.row_bytes + v * 16) =
                  reinterpret_cast<const int4*>(newrow)[v];
        }
      } else if (pull) {
        wrote = m > 0;
        const long long total = (long long)m * rvec;
        constexpr int U = 8;   // host reads in flight per thread
        for (long long e0 = tid; e0 < total; e0 += (long long)U * NT) {
          int4 v[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const long long e = e0 + (long long)u * NT;
            if (e < total) {
              const int qq = (int)(e / rvec);
              const int cidx = (int)(e - (long long)qq * rvec);
              if (miss_i[qq] & HS_SLOT_MISS_FLAG) continue;   // a follower's own new token
              const int pos = sel[miss_i[qq]];
              v[u] = (pass == 0 && appended && pos == len)
                         ? reinterpret_cast<const int4*>(newrow)[cidx]
                         : *reinterpret_cast<const int4*>(src_base + (size_t)pos * g.row_bytes + cidx * 16);
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const long long e = e0 + (long long)u * NT;
            if (e < total) {
              const int qq = (int)(e / rvec);
              const int cidx = (int)(e - (long long)qq * rvec);
              if (miss_i[qq] & HS_SLOT_MISS_FLAG) continue;
              *reinterpret_cast<int4*>(dst_base + (size_t)victim[qq] * g.row_bytes + cidx * 16) = v[u];
            }
          }
        }
      } else if (pass == 0 && appended && m > 0 && sel[miss_i[m - 1] & ~HS_SLOT_MISS_FLAG] == len) {
        // the appended token is the highest position: if it missed, it is the last miss
        wrote = true;
        for (int v = tid; v < rvec; v += NT)
          *reinterpret_cast<int4*>(dst_base + (size_t)victim[m - 1] * g.row_bytes + v * 16) =
              reinterpret_cast<const int4*>(newrow)[v];
      }
      if (wrote) fence_proxy_async_global();   // generic-proxy slot writes, read by bulk copies
    }
    // ======================= 4. publication =======================
    __syncthreads();
    HS_TRACE_IF(p, 1, 7, tid == 0 && pass == 0 && ri == (int)blockIdx.x);
    // every thread's writes for this request (ordered before thread 0 by the
    // barrier above) are made visible GPU-wide by a full fence before the release
    // store that the attention kernel's acquire load pairs with (the release
    // store alone measured far slower on some machines)
    if (pass == 0 && p.publish && tid == 0) {
      __threadfence();
      if (!(p.fault == 1 && ri == 0)) st_release(p.s.ready + ri, (unsigned)kkr + 1u);   // rows + 1
    }
    HS_TRACE_IF(p, 1, 16, tid == 0 && pass == 0 && ri == (int)blockIdx.x);

    HS_TRACE_IF(p, 1, 12, tid == 0 && pass == 0 && ri == (int)blockIdx.x);
    // the next threshold to the exact key of rank k_next: the low digit of that
    // key from a histogram of the keys with its high digit (the candidates when
    // they hold every key that large, else all keys); off the critical path
    if (pass == 0 && sh.thr_src != 0 && N <= CAND_MAX_N_PER_K * K) {
      const int src = sh.thr_src;
      const uint32_t bt = (uint32_t)sh.bt;
      for (int c = tid; c < IDX_BINS / 4; c += NT) reinterpret_cast<uint4*>(h)[c] = make_uint4(0, 0, 0, 0);
      __syncthreads();
      if (src == 1) {
        const uint2* cl = p.s.cand + (long long)ri * 2 * KR;
        const int cnt = min(sh.cnt, 2 * KR);
        for (int i = tid; i < cnt; i += NT) {
          const uint32_t k = __ldcg(cl + i).y;
          if ((k >> 12) == bt) atomicAdd(&h[k & 4095u], 1u);
        }
      } else {
        const uint32_t* keys = p.s.scores + (long long)ri * p.score_stride;
        for (int i = tid; i < N; i += NT) {
          const uint32_t k = __ldcg(keys + i);
          if ((k >> 12) == bt) atomicAdd(&h[k & 4095u], 1u);
        }
      }
      __syncthreads();
      select_digit(h, k_next - sh.above_t, sh.scan, &sh.b2, &sh.above2);
      if (tid == 0) sh.thr_next = (bt << 12) | (uint32_t)sh.b2;
    }

    HS_TRACE_IF(p, 1, 13, tid == 0 && pass == 0 && ri == (int)blockIdx.x);
    // ======================= 5. metadata after publication =======================
    // LRU and random: every used slot is refreshed; FIFO: only the filled ones (used == 2)
    const bool fifo = p.replacement == HS_REPLACE_FIFO;
    auto refreshed = [&](uint8_t u) { return fifo ? u == 2 : u != 0; };
    if (kx > 0) {
      for (int i = tid; i < kx; i += NT) {
        const int sl = slot_sel[i];
        if (refreshed(used[sl])) stamp[sl] = t;
      }
      // new list: slots not refreshed keep their order, refreshed slots (all with
      // the newest stamp) go last by slot
      // (the same warp segments as above: the list's entries and the slots)
      int nu = 0, nus = 0;
      for (int j = wj0; j < wj1; j += 32) {
        const int jj = j + lane;
        nu += __popc(__ballot_sync(FULL_MASK, jj < wj1 && !refreshed(used[ord[jj]])));
        nus += __popc(__ballot_sync(FULL_MASK, jj < wj1 && refreshed(used[jj])));
      }
      int n_unused;
      const int2 un = block_exclusive_scan2<NT>(lane == 0 ? nu : 0, lane == 0 ? nus : 0, sh.scan, &n_unused, nullptr);
      int ub = __shfl_sync(FULL_MASK, un.x, 0);
      int sb = n_unused + __shfl_sync(FULL_MASK, un.y, 0);
      for (int j = wj0; j < wj1; j += 32) {
        const int jj = j + lane;
        const int sl = jj < wj1 ? ord[jj] : 0;
        const bool keep = jj < wj1 && !refreshed(used[sl]);
        const unsigned bk = __ballot_sync(FULL_MASK, keep);
        if (keep) order[ub + __popc(bk & lt)] = sl;
        ub += __popc(bk);
        const bool rf = jj < wj1 && refreshed(used[jj]);
        const unsigned br = __ballot_sync(FULL_MASK, rf);
        if (rf) order[sb + __popc(br & lt)] = jj;
        sb += __popc(br);
      }
      if (tid == 0) {
        p.s.step[rlx] = t + 1;
        // counters of the selected positions (an allocated new token is neither)
        red_add_u64(&p.s.hits[rlx], (unsigned long long)(kk - (m - extra)));
        red_add_u64(&p.s.misses[rlx], (unsigned long long)(m - extra));
        // rows over the host link: page mode, every row of a missed page below the length
        const int mrows = !paged ? m - extra
                                 : m * PS - ((m > 0 && sel[miss_i[m - 1] & ~HS_SLOT_MISS_FLAG] == N - 1) ? N * PS - Np : 0);
        red_add_u64(&p.s.glob[0], (unsigned long long)mrows * g.row_bytes);
      }
    }
    if (pass > 0 && tid == 0) p.s.sh_armed[rlx] = 1;   // ready for the follower's call
    }   // passes
    if (sel_out)
      for (int i = tid; i < KR; i += NT) sel_out[i] = i < kkr ? row_pos(i) : -1;
    if (skip_rest) {
      __syncthreads();
      continue;
    }
    // a group lead that does not prefetch leaves the selection for its followers
    if (p.role == ROLE_SELECT && !p.share_prefetch && p.n_follow > 0 && sh.ok) {
      for (int f = 1; f <= p.n_follow; ++f) {
        int32_t* fp = p.s.sh_sel + (rl + f) * KR;
        for (int i = tid; i < kk; i += NT) fp[i] = sel[i];
        if (tid == 0) {
          p.s.sh_kk[rl + f] = kk;
          p.s.sh_armed[rl + f] = 1;
        }
      }
    }

    HS_TRACE_IF(p, 1, 14, tid == 0 && ri == (int)blockIdx.x);
    // the appended token: key to the HBM store, row to the pinned host copy
    if (appended) {
      const int rvec = g.row_bytes / 16;
      int4* dst = reinterpret_cast<int4*>(p.s.host_kv + (rl * g.max_context + len) * g.row_elems);
      for (int v = tid; v < rvec; v += NT) dst[v] = reinterpret_cast<const int4*>(newrow)[v];
      if (tid < g.d_idx / 16)
        reinterpret_cast<int4*>(p.s.idx_keys + (rl * g.max_context + len) * g.d_idx)[tid] =
            reinterpret_cast<const int4*>(newkey)[tid];
      // page mode: its page's bounds take the new key (a page it opens: the key alone)
      const int hk = g.d_idx / 16;
      if (paged && tid < 2 * hk) {
        int4* bd = reinterpret_cast<int4*>(p.s.pbound + (rl * g.max_pages + (len >> psh)) * 2 * g.d_idx);
        const bool hi = tid < hk;
        const int4 kn = reinterpret_cast<const int4*>(newkey)[hi ? tid : tid - hk];
        if ((len & (PS - 1)) == 0) bd[tid] = kn;
        else bd[tid] = hi ? vmax16(bd[tid], kn) : vmin16(bd[tid], kn);
      }
    }
    HS_TRACE_IF(p, 1, 15, tid == 0 && ri == (int)blockIdx.x);
    // lengths and thresholds: only once every CTA of the launch has read them
    if (tid == 0) {
      if (!wait_counter(&p.s.sync[0], (unsigned)(p.sel_grid - p.n_resolvers))) {
        set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
      } else {
        if (appended) {
          p.s.length[rl] = Np;
          red_add_u64(&p.s.glob[1], (unsigned long long)g.row_bytes);
        }
        if (sh.ok) p.s.cand_thr[rl] = sh.thr_next;
      }
    }
    __syncthreads();
    HS_TRACE_IF(p, 1, 8, tid == 0 && ri == (int)blockIdx.x);
  }
  // the last resolver to finish resets the launch's shared counters (once every
  // scorer CTA has counted itself in)
  if (tid == 0) {
    const unsigned prev = atom_acq_rel_add(&p.s.sync[1], 1u);
    if (prev + 1 == (unsigned)p.n_resolvers) {
      if (!wait_counter(&p.s.sync[0], (unsigned)(p.sel_grid - p.n_resolvers)))
        set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
      p.s.sync[0] = 0;
      p.s.sync[1] = 0;
    }
  }
}

template <int NCH, int NH, bool PG = false>
static cudaError_t run_select(const DecodeParams* p, size_t smem, cudaStream_t st) {
  auto kern = select_kernel<NCH, NH, PG>;
  if (p == nullptr) return allow_smem(kern, smem);
  return launch_pdl(kern, dim3(p->sel_grid), dim3(NT), smem, st, *p);
}

// single-head indexer: d_idx 16..256; the multi-head indexer: d_idx 64 or 128,
// 2, 4 or 8 heads; page mode: unit rows of 2 * d_idx bytes (d_idx 64 or 128)
static cudaError_t dispatch_select(const Geometry& g, const DecodeParams* p, size_t smem, cudaStream_t st) {
  if (g.page_shift > 0) {
    switch (g.d_idx) {
      case 64: return run_select<8, 1, true>(p, smem, st);
      case 128: return run_select<16, 1, true>(p, smem, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (g.idx_heads <= 1) {
    switch (g.d_idx) {
      case 16: return run_select<1, 1>(p, smem, st);
      case 32: return run_select<2, 1>(p, smem, st);
      case 64: return run_select<4, 1>(p, smem, st);
      case 128: return run_select<8, 1>(p, smem, st);
      case 256: return run_select<16, 1>(p, smem, st);
      default: return cudaErrorInvalidValue;
    }
  }
  const int key = g.d_idx * 16 + g.idx_heads;
  switch (key) {
    case 64 * 16 + 2: return run_select<4, 2>(p, smem, st);
    case 64 * 16 + 4: return run_select<4, 4>(p, smem, st);
    case 64 * 16 + 8: return run_select<4, 8>(p, smem, st);
    case 128 * 16 + 2: return run_select<8, 2>(p, smem, st);
    case 128 * 16 + 4: return run_select<8, 4>(p, smem, st);
    case 128 * 16 + 8: return run_select<8, 8>(p, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t prepare_select(const Geometry& g, size_t smem) { return dispatch_select(g, nullptr, smem, 0); }

cudaError_t launch_select(const DecodeParams& p, size_t smem, cudaStream_t st) {
  return dispatch_select(p.g, &p, smem, st);
}

}  // namespace hs

// ===========================================================================
// A follower layer's call under a shared selection whose group lead already
// resolved it (share_prefetch): no scoring, no top-k, no RESOLVE.  One CTA per
// request appends this layer's token (key to the HBM store, row to the host
// copy, length + 1), puts that row into its slot when the shared selection took
// it (the lead could not: the row did not exist yet), and publishes the
// prepared slots to the attention kernel launched after it.
// ===========================================================================
namespace hs {

constexpr int FOL_THREADS = 256;

__global__ void __launch_bounds__(FOL_THREADS) follow_kernel(DecodeParams p) {
  const Geometry& g = p.g;
  const int tid = threadIdx.x;
  const int ri = blockIdx.x;
  const int K = g.top_k;
  __shared__ int s_kk, s_len, s_ok;
  griddep_wait();   // the lead's slots, lengths and earlier appends
  griddep_launch_dependents();
  int32_t* sel_out = p.sel_out ? p.sel_out + (long long)ri * K : nullptr;
  const int req = p.req_ids ? p.req_ids[ri] : ri;
  if (req < 0 || req >= g.max_requests) {
    if (tid == 0) {
      set_error(p.s.dev_error, HS_DEVERR_REQ_RANGE);
      __threadfence();
      st_release(p.s.ready + ri, 1u);   // nothing selected
    }
    if (sel_out)
      for (int i = tid; i < K; i += FOL_THREADS) sel_out[i] = -1;
    return;
  }
  const long long rl = (long long)req * g.n_layers + p.layer;
  if (tid == 0) {
    const int len = p.s.length[rl];
    int N = len;
    if (p.new_kv) {
      if (len + 1 <= g.max_context) N = len + 1;
      else set_error(p.s.dev_error, HS_DEVERR_CAPACITY);
    }
    const int kk = p.s.sh_kk[rl];
    const bool ok = p.s.sh_armed[rl] != 0 && kk == min(K, N);
    if (!ok) set_error(p.s.dev_error, HS_DEVERR_NO_LEAD);
    p.s.sh_armed[rl] = 0;
    s_kk = ok ? kk : 0;
    s_len = len;
    s_ok = N > len;   // appended
  }
  __syncthreads();
  const int kk = s_kk, len = s_len;
  const bool appended = s_ok != 0;
  const int rvec = g.row_bytes / 16;
  // this layer's token: into its slot when the shared selection took it
  const int pend = kk > 0 ? p.s.sh_pend[rl] : -1;
  if (appended && pend >= 0 && pend < g.hot_slots) {
    const int4* src = reinterpret_cast<const int4*>(p.new_kv + (long long)ri * g.row_elems);
    int4* dst = reinterpret_cast<int4*>(p.s.hot + ((size_t)rl * g.hot_slots + pend) * g.row_elems);
    for (int v = tid; v < rvec; v += FOL_THREADS) dst[v] = src[v];
  }
  // the prepared slots and the selection, for the attention kernel and sel_out
  const int32_t* fs = p.s.sh_slots + rl * K;
  const int32_t* fp = p.s.sh_sel + rl * K;
  int32_t* sos = p.s.slot_of_sel + (long long)ri * K;
  int32_t* sel_g = p.s.sel + (long long)ri * K;
  for (int i = tid; i < K; i += FOL_THREADS) {
    const int pos = i < kk ? __ldcg(fp + i) : -1;
    if (i < kk) {
      sos[i] = __ldcg(fs + i);
      sel_g[i] = pos;
    }
    if (sel_out) sel_out[i] = pos;
  }
  // the append itself: key to the HBM store, row to the pinned host copy
  if (appended) {
    const int4* src = reinterpret_cast<const int4*>(p.new_kv + (long long)ri * g.row_elems);
    int4* dst = reinterpret_cast<int4*>(p.s.host_kv + ((size_t)rl * g.max_context + len) * g.row_elems);
    for (int v = tid; v < rvec; v += FOL_THREADS) dst[v] = src[v];
    if (tid < g.d_idx / 16)
      reinterpret_cast<int4*>(p.s.idx_keys + ((size_t)rl * g.max_context + len) * g.d_idx)[tid] =
          reinterpret_cast<const int4*>(p.new_keys + (long long)ri * g.d_idx)[tid];
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");   // slot writes, read by bulk copies
  __syncthreads();
  if (tid == 0) {
    if (appended) {
      p.s.length[rl] = len + 1;
      red_add_u64(&p.s.glob[1], (unsigned long long)g.row_bytes);
    }
    __threadfence();
    st_release(p.s.ready + ri, (unsigned)kk + 1u);   // k_eff + 1
  }
}

cudaError_t launch_follow(const DecodeParams& p, cudaStream_t st) {
  return launch_pdl(follow_kernel, dim3(p.n_req), dim3(FOL_THREADS), 0, st, p);
}

}  // namespace hs
