// Indexer scores: s[p] = sum_j q_idx[j] * K_idx[p][j] for every position of
// every request that needs a selection (more positions than k), as 24-bit
// order-preserving keys, plus a 4096-bin histogram of the keys' high 12 bits
// per request (the first digit of the exact top-k select that follows).
//
// Method: "10月14日学习笔记" (zgchen.com), "HiSparse / 动机": an indexer scores
// the context and attention runs over the top-k tokens only.  The score is an
// int8 query dotted with each position's int8 index key, summed exactly in
// int32 with dp4a.
//
// Design (sm_103a), HBM-bound (d_idx bytes read per position, 4 written):
//  * Persistent grid, one CTA per SM.  The positions of all requests are
//    flattened and split into equal contiguous ranges, one per CTA (so every CTA
//    streams the same number of bytes); a CTA meets at most a few request
//    boundaries.  A per-request table in shared memory (position prefix, request
//    id, length) locates every tile without global loads.
//  * Thread 0 streams the range HBM -> shared memory as tiles of up to
//    IDX_TILE_BYTES (cut at request boundaries) with 1-D bulk async copies
//    (cp.async.bulk, mbarrier completion), up to six stages deep: with one tile
//    being scored the rest keep >= 128 KB per SM in flight, which is what a
//    single CTA per SM needs to reach full HBM bandwidth on this part.
//  * One lane per position.  Lane l reads the 16-byte chunks of its position in
//    the rotated order (c + rot) mod NCH so the 8 lanes of a quarter warp hit 8
//    different bank groups; the query chunks sit in registers in the same rotated
//    order, so the rotation costs nothing in the inner loop.
//  * key = score + 2^22 (|score| <= 128*128*256 = 2^22) is stored to a per-call
//    scratch row; the high-digit histogram is kept in shared memory per request
//    segment and added to the request's global histogram when the segment ends.
//  * Keys at or above the request's candidate threshold (set by the previous
//    call's top-k) are also appended, with their positions, to a short
//    per-request list (ballot + popcount into per-warp shared-memory buffers,
//    one global atomic per flush), which lets the top-k skip the full scan when
//    the selection moved little since the previous step; requests without a
//    threshold take a separate loop that does none of this.
//  * Launched as a programmatic dependent: barrier and histogram set-up overlap
//    the previous kernel's tail.
#include "hs_internal.cuh"

namespace hs {

namespace {

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int SC_MAX_STAGES = 6;
constexpr size_t SC_SMEM_LIMIT = 227 * 1024;

constexpr int SC_CBUF = 1024;   // candidates buffered per CTA before a flush to the request's list
constexpr int SC_WBUF = SC_CBUF / (SC_THREADS / 32);   // per warp

struct ScoreLayout {
  size_t bar, pprefix, req, len, thr, hist, cbuf, stage, total;
  int nstage;
};

__host__ __device__ inline ScoreLayout score_layout(const Geometry& g) {
  ScoreLayout L;
  size_t off = 0;
  L.bar = off;
  off += 128;
  L.pprefix = off;   // long long [n + 1]: first flattened position of request i
  off += align_up((size_t)(g.max_requests + 1) * 8, 128);
  L.req = off;       // int [n]: request id (-1: no selection needed)
  off += align_up((size_t)g.max_requests * 4, 128);
  L.len = off;       // int [n]: positions of request i this call (with the appended token)
  off += align_up((size_t)g.max_requests * 4, 128);
  L.thr = off;       // u32 [n]: candidate threshold of request i (0: list nothing)
  off += align_up((size_t)g.max_requests * 4, 128);
  L.hist = off;
  off += IDX_BINS * 4;
  L.cbuf = off;     // uint2 [SC_CBUF]: (position, key) listed since the last flush
  off += (size_t)SC_CBUF * 8;
  L.stage = off;
  // as many 32 KB stages as fit (at least two): with one stage being scored,
  // the others keep >= 128 KB of copies in flight per SM
  const size_t room = SC_SMEM_LIMIT > off ? (SC_SMEM_LIMIT - off) / IDX_TILE_BYTES : 0;
  L.nstage = (int)(room < 2 ? 2 : (room > SC_MAX_STAGES ? SC_MAX_STAGES : room));
  off += (size_t)L.nstage * IDX_TILE_BYTES;
  L.total = off;
  return L;
}

}  // namespace

size_t score_smem_bytes(const Geometry& g) { return score_layout(g).total; }

template <int NCH>
__global__ void __launch_bounds__(SC_THREADS) score_kernel(DecodeParams p) {
  constexpr int d = NCH * 16;
  constexpr int TP = IDX_TILE_BYTES / d;   // positions per full tile
  const Geometry& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31;
  const int c = blockIdx.x;
  const int K = g.top_k;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  const ScoreLayout L = score_layout(g);
  const int NST = L.nstage;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + L.bar);
  long long* pprefix = reinterpret_cast<long long*>(smem_raw + L.pprefix);
  int* req_s = reinterpret_cast<int*>(smem_raw + L.req);
  int* len_s = reinterpret_cast<int*>(smem_raw + L.len);
  uint32_t* thr_s = reinterpret_cast<uint32_t*>(smem_raw + L.thr);
  uint2* cbuf = reinterpret_cast<uint2*>(smem_raw + L.cbuf);
  __shared__ int cb_wn[SC_THREADS / 32], cb_base;
  const int warp = tid >> 5;
  uint2* wbuf = cbuf + warp * SC_WBUF;   // this warp's part of the buffer
  int wn = 0;                            // entries in it (warp-uniform)
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw + L.hist);
  unsigned char* stage = smem_raw + L.stage;
  __shared__ long long scan_tmp[SC_THREADS / 32 + 1];
  __shared__ __align__(16) unsigned char new_key[256];
  HS_TRACE(p, 0, 0);

  for (int b = tid; b < IDX_BINS; b += SC_THREADS) hist[b] = 0;
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  griddep_wait();   // lengths, keys and the query come from earlier stream work
  griddep_launch_dependents();

  // ---- positions of every request that needs a selection (N > k) ----------------
  long long carry = 0;
  for (int base = 0; base < p.n_req; base += SC_THREADS) {
    const int i = base + tid;
    long long npos = 0;
    if (i < p.n_req) {
      const int req = p.req_ids ? p.req_ids[i] : i;
      int N = 0;
      if (req >= 0 && req < g.max_requests) {
        N = p.s.length[(long long)req * g.n_layers + p.layer];
        if (p.new_kv && N + 1 <= g.max_context) ++N;   // the token this call appends
      }
      npos = N > K ? N : 0;
      req_s[i] = npos ? req : -1;
      len_s[i] = N;
      thr_s[i] = (npos && p.s.cand_thr) ? p.s.cand_thr[(long long)req * g.n_layers + p.layer] : 0u;
      if (c == 0 && p.s.call_n) p.s.call_n[i] = N;   // for RESOLVE's view of the attention split
    }
    // block-wide exclusive scan of 64-bit counts
    long long incl = npos;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long n = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) scan_tmp[tid >> 5] = incl;
    __syncthreads();
    if (tid < 32) {
      long long x = tid < SC_THREADS / 32 ? scan_tmp[tid] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(FULL_MASK, x, o);
        if (lane >= o) x += n;
      }
      if (tid < SC_THREADS / 32) scan_tmp[tid] = x;   // inclusive warp totals
    }
    __syncthreads();
    const long long wbase = (tid >> 5) ? scan_tmp[(tid >> 5) - 1] : 0;
    if (i < p.n_req) pprefix[i] = carry + wbase + incl - npos;
    carry += scan_tmp[SC_THREADS / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) pprefix[p.n_req] = carry;
  __syncthreads();
  HS_TRACE(p, 0, 1);
  const long long P = carry;
  if (P == 0) return;
  const int Gc = (int)min((long long)gridDim.x, (P + TP - 1) / TP);
  if (c >= Gc) return;
  const long long a0 = (long long)c * P / Gc, a1 = (long long)(c + 1) * P / Gc;
  int r0 = 0;
  {
    int lo = 0, hi = p.n_req - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pprefix[mid] <= a0) lo = mid;
      else hi = mid - 1;
    }
    r0 = lo;
    while (pprefix[r0 + 1] <= a0) ++r0;
  }

  // Tiles: consecutive pieces of [a0, a1), at most TP positions, never across a
  // request boundary.  Walking them needs only the shared tables.
  struct Cursor {
    int r;
    long long a;   // flattened position of the next tile
  };
  struct TileRef {
    int r, npos, newpos;   // newpos: position of the appended token (its key comes from the input), or -1
    long long pos0, rl;
  };
  auto next_tile = [&](Cursor& cu) -> TileRef {
    while (pprefix[cu.r + 1] <= cu.a) ++cu.r;
    TileRef tr;
    tr.r = cu.r;
    tr.rl = (long long)req_s[cu.r] * g.n_layers + p.layer;
    const int N = len_s[cu.r];
    tr.newpos = p.new_kv ? N - 1 : -1;
    tr.pos0 = cu.a - pprefix[cu.r];
    tr.npos = (int)min(min((long long)TP, (long long)N - tr.pos0), a1 - cu.a);
    cu.a += tr.npos;
    return tr;
  };
  // tile count of this CTA
  int ntile = 0;
  {
    Cursor cu{r0, a0};
    while (cu.a < a1) {
      (void)next_tile(cu);
      ++ntile;
    }
  }

  Cursor cu_issue{r0, a0};
  const uint64_t stream_policy = l2_evict_first_policy();   // index keys are read once per call
  auto issue = [&](int k) {   // tile k into stage k % NST
    const TileRef tr = next_tile(cu_issue);
    const int s = k % NST;
    const uint32_t bytes = (uint32_t)(tr.npos * d);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&bar[s], bytes);
    bulk_g2s_hint(stage + (size_t)s * IDX_TILE_BYTES, p.s.idx_keys + (tr.rl * g.max_context + tr.pos0) * d, bytes,
                  &bar[s], stream_policy);
  };
  if (tid == 0)
    for (int k = 0; k < NST && k < ntile; ++k) issue(k);

  const int rot = NCH >= 8 ? (lane & (NCH - 1)) : ((lane & 7) / (8 / NCH));
  int4 qrot[NCH];
  int q_r = -1;

  Cursor cu{r0, a0};
  bool timed_out = false;
  int consumed = 0;
  for (int k = 0; k < ntile; ++k) {
    const int s = k % NST;
    const TileRef tr = next_tile(cu);
    if (tr.r != q_r) {   // the request's query chunks, rotated per lane
      q_r = tr.r;
      const int4* qsrc = reinterpret_cast<const int4*>(p.q_idx + (long long)tr.r * d);
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) qrot[cc] = qsrc[(cc + rot) & (NCH - 1)];
    }
    const int jnew = (tr.newpos >= tr.pos0 && tr.newpos < tr.pos0 + tr.npos) ? (int)(tr.newpos - tr.pos0) : -1;
    if (jnew >= 0 && tid < NCH)   // the appended token's key is not in the store yet
      reinterpret_cast<int4*>(new_key)[tid] = reinterpret_cast<const int4*>(p.new_keys + (long long)tr.r * d)[tid];
    const bool ok = mbar_wait_bounded(&bar[s], (uint32_t)((k / NST) & 1));
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    consumed = k + 1;
    HS_TRACE_IF(p, 0, 2, tid == 0 && k == 0);
    const unsigned char* tile = stage + (size_t)s * IDX_TILE_BYTES;
    uint32_t* keys_out = p.s.scores + (long long)tr.r * p.score_stride + tr.pos0;
    const uint32_t thr = thr_s[tr.r];   // block-uniform
    // one position per thread and pass: dp4a over the 16-byte chunks in the
    // lane's rotated order; key = score + 2^22
    auto score_at = [&](int j) -> uint32_t {
      const unsigned char* rowp = j == jnew ? new_key : tile + j * d;
      int acc = 0;
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int4 kv = *reinterpret_cast<const int4*>(rowp + (((cc + rot) & (NCH - 1)) << 4));
        acc = __dp4a(kv.x, qrot[cc].x, acc);
        acc = __dp4a(kv.y, qrot[cc].y, acc);
        acc = __dp4a(kv.z, qrot[cc].z, acc);
        acc = __dp4a(kv.w, qrot[cc].w, acc);
      }
      return (uint32_t)(acc + IDX_KEY_BIAS);
    };
    if (thr == 0u) {   // no listing for this request (kept as a separate, lean loop)
      for (int j = tid; j < tr.npos; j += SC_THREADS) {
        const uint32_t key = score_at(j);
        keys_out[j] = key;
        atomicAdd(&hist[key >> 12], 1u);
      }
    } else {
      for (int j0 = 0; j0 < tr.npos; j0 += SC_THREADS) {
        const int j = j0 + tid;
        uint32_t key = 0;
        if (j < tr.npos) {
          key = score_at(j);
          keys_out[j] = key;
          atomicAdd(&hist[key >> 12], 1u);
        }
        // buffer the keys at or above the threshold (per warp, no atomics)
        const bool c = j < tr.npos && key >= thr;
        const unsigned m = __ballot_sync(FULL_MASK, c);
        if (m) {
          const int at = wn + __popc(m & ((1u << lane) - 1u));
          const uint2 v = make_uint2((uint32_t)(tr.pos0 + j), key);
          if (wn + __popc(m) <= SC_WBUF) {
            if (c) wbuf[at] = v;
            wn += __popc(m);
          } else if (c) {   // this warp's part is full (narrow keys): straight to the list
            const unsigned g2 = atomicAdd(p.s.cand_cnt + tr.r, 1u);
            if (g2 < 2u * (unsigned)K) p.s.cand[(long long)tr.r * 2 * K + g2] = v;
          }
        }
      }
    }
    // stage s consumed; histogram updates of this tile done; is any warp's buffer
    // too full for another tile?
    bool near_full = false;
    if (thr == 0u) __syncthreads();
    else near_full = __syncthreads_or(wn + 32 * ((TP + SC_THREADS - 1) / SC_THREADS) > SC_WBUF);
    if (tid == 0 && k + NST < ntile) issue(k + NST);
    // end of this request's segment: add the histogram to the request's one
    const bool seg_end = (k + 1 == ntile) || (pprefix[tr.r + 1] <= cu.a);
    if (thr != 0u && (seg_end || near_full)) {   // flush the listed keys (one global atomic)
      if (lane == 0) cb_wn[warp] = wn;
      __syncthreads();
      if (tid == 0) {
        int n = 0;
        for (int w2 = 0; w2 < SC_THREADS / 32; ++w2) n += cb_wn[w2];
        cb_base = n ? (int)atomicAdd(p.s.cand_cnt + tr.r, (unsigned)n) : 0;
      }
      __syncthreads();
      int off = cb_base;
      for (int w2 = 0; w2 < warp; ++w2) off += cb_wn[w2];
      uint2* dst = p.s.cand + (long long)tr.r * 2 * K;
      for (int i = lane; i < wn; i += 32)
        if (off + i < 2 * K) dst[off + i] = wbuf[i];
      wn = 0;
      __syncthreads();   // cb_wn and the buffer are reused
    }
    if (seg_end) {
      uint32_t* gh = p.s.hist + (long long)tr.r * IDX_BINS;
      for (int b = tid; b < IDX_BINS; b += SC_THREADS) {
        const uint32_t v = hist[b];
        if (v) {
          atomicAdd(&gh[b], v);
          hist[b] = 0;
        }
      }
      __syncthreads();
    }
  }
  HS_TRACE(p, 0, 3);
  if (timed_out) {
    if (tid == 0) {
      const int issued = min(ntile, consumed + NST);
      for (int k = consumed; k < issued; ++k)
        (void)mbar_wait_bounded(&bar[k % NST], (uint32_t)((k / NST) & 1));
      set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
    }
    __syncthreads();
  }
}

template <int NCH>
static cudaError_t run_score(const DecodeParams* p, size_t smem, cudaStream_t st) {
  auto kern = score_kernel<NCH>;
  if (p == nullptr) return allow_smem(kern, smem);
  return launch_pdl(kern, dim3(p->score_grid), dim3(SC_THREADS), smem, st, *p);
}

static cudaError_t dispatch_score(int d_idx, const DecodeParams* p, size_t smem, cudaStream_t st) {
  switch (d_idx) {
    case 16: return run_score<1>(p, smem, st);
    case 32: return run_score<2>(p, smem, st);
    case 64: return run_score<4>(p, smem, st);
    case 128: return run_score<8>(p, smem, st);
    case 256: return run_score<16>(p, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t prepare_score(const Geometry& g, size_t smem) { return dispatch_score(g.d_idx, nullptr, smem, 0); }

cudaError_t launch_score(const DecodeParams& p, size_t smem, cudaStream_t st) {
  return dispatch_score(p.g.d_idx, &p, smem, st);
}

}  // namespace hs
