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
//  * Persistent grid (SMs x 2).  The positions of all requests are flattened
//    into tiles of IDX_TILE_BYTES of keys; CTA c takes a contiguous tile range,
//    so it meets at most a few request boundaries.
//  * Thread 0 streams the tiles HBM -> shared memory with 1-D bulk async copies
//    (cp.async.bulk, mbarrier completion), IDX_STAGES deep.
//  * One lane per position.  Lane l reads the 16-byte chunks of its position in
//    the rotated order (c + rot) mod NCH so the 8 lanes of a quarter warp hit 8
//    different bank groups; the query chunks sit in registers in the same rotated
//    order, so the rotation costs nothing in the inner loop.
//  * key = score + 2^22 (|score| <= 128*128*256 = 2^22) is stored to a per-call
//    scratch row; the high-digit histogram is kept in shared memory per request
//    segment and added to the request's global histogram when the segment ends.
#include "hs_internal.cuh"

namespace hs {

namespace {

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct ScoreLayout {
  size_t bar, prefix, hist, stage, total;
};

__host__ __device__ inline ScoreLayout score_layout(const Geometry& g) {
  ScoreLayout L;
  size_t off = 0;
  L.bar = off;
  off += 128;
  L.prefix = off;
  off += align_up((size_t)(g.max_requests + 1) * 4, 128);
  L.hist = off;
  off += IDX_BINS * 4;
  L.stage = off;
  off += (size_t)IDX_STAGES * IDX_TILE_BYTES;
  L.total = off;
  return L;
}

}  // namespace

size_t score_smem_bytes(const Geometry& g) { return score_layout(g).total; }

template <int NCH>
__global__ void __launch_bounds__(SC_THREADS) score_kernel(DecodeParams p) {
  constexpr int d = NCH * 16;
  constexpr int TP = IDX_TILE_BYTES / d;   // positions per tile
  const Geometry& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31;
  const int c = blockIdx.x;
  const int K = g.top_k;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  const ScoreLayout L = score_layout(g);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + L.bar);
  int* prefix = reinterpret_cast<int*>(smem_raw + L.prefix);   // first tile of request i
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw + L.hist);
  unsigned char* stage = smem_raw + L.stage;
  __shared__ int scan_tmp[SC_THREADS / 32 + 1];
  HS_TRACE(p, 0, 0);

  // ---- tiles of every request that needs a selection (N > k) ------------------
  int carry = 0;
  for (int base = 0; base < p.n_req; base += SC_THREADS) {
    const int i = base + tid;
    int tiles = 0;
    if (i < p.n_req) {
      const int req = p.req_ids ? p.req_ids[i] : i;
      if (req >= 0 && req < g.max_requests) {
        int N = p.s.length[(long long)req * g.n_layers + p.layer];
        if (p.new_kv && N + 1 <= g.max_context) ++N;   // the token this call appends
        if (N > K) tiles = (N + TP - 1) / TP;
      }
    }
    int tot;
    const int ex = block_exclusive_scan<SC_THREADS>(tiles, scan_tmp, &tot);
    if (i < p.n_req) prefix[i] = carry + ex;
    carry += tot;
  }
  for (int b = tid; b < IDX_BINS; b += SC_THREADS) hist[b] = 0;
  if (tid == 0) {
    prefix[p.n_req] = carry;
    for (int s = 0; s < IDX_STAGES; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  HS_TRACE(p, 0, 1);
  const long long T = carry;
  if (T == 0) return;
  const int Gc = (int)min((long long)gridDim.x, T);
  if (c >= Gc) return;
  const int t0 = (int)((long long)c * T / Gc), t1 = (int)((long long)(c + 1) * T / Gc);
  int r0 = 0;
  {
    int lo = 0, hi = p.n_req - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= t0) lo = mid;
      else hi = mid - 1;
    }
    r0 = lo;
    while (prefix[r0 + 1] <= t0) ++r0;
  }

  // where tile t of this CTA lives
  struct TileRef {
    int r, npos, newpos;   // newpos: position of the appended token (its key comes from the input), or -1
    long long pos0, rl;
  };
  auto tile_ref = [&](int t, int& rc) -> TileRef {
    while (prefix[rc + 1] <= t) ++rc;
    TileRef tr;
    tr.r = rc;
    const int req = p.req_ids ? p.req_ids[rc] : rc;
    tr.rl = (long long)req * g.n_layers + p.layer;
    int N = p.s.length[tr.rl];
    tr.newpos = -1;
    if (p.new_kv && N + 1 <= g.max_context) tr.newpos = N++;
    tr.pos0 = (long long)(t - prefix[rc]) * TP;
    tr.npos = (int)min((long long)TP, N - tr.pos0);
    return tr;
  };

  int r_issue = r0;
  auto issue = [&](int k) {   // tile t0 + k into stage k % IDX_STAGES
    const TileRef tr = tile_ref(t0 + k, r_issue);
    const int s = k % IDX_STAGES;
    const uint32_t bytes = (uint32_t)(tr.npos * d);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&bar[s], bytes);
    bulk_g2s(stage + (size_t)s * IDX_TILE_BYTES, p.s.idx_keys + (tr.rl * g.max_context + tr.pos0) * d, bytes,
             &bar[s]);
  };
  const int ntile = t1 - t0;
  if (tid == 0)
    for (int k = 0; k < IDX_STAGES && k < ntile; ++k) issue(k);

  const int rot = NCH >= 8 ? (lane & (NCH - 1)) : ((lane & 7) / (8 / NCH));
  int4 qrot[NCH];
  int q_r = -1;
  __shared__ __align__(16) unsigned char new_key[256];

  int r_cur = r0;
  bool timed_out = false;
  int consumed = 0;
  for (int k = 0; k < ntile; ++k) {
    const int s = k % IDX_STAGES;
    const TileRef tr = tile_ref(t0 + k, r_cur);
    if (tr.r != q_r) {   // the request's query chunks, rotated per lane
      q_r = tr.r;
      const int4* qsrc = reinterpret_cast<const int4*>(p.q_idx + (long long)tr.r * d);
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) qrot[cc] = qsrc[(cc + rot) & (NCH - 1)];
    }
    const int jnew = (tr.newpos >= tr.pos0 && tr.newpos < tr.pos0 + tr.npos) ? (int)(tr.newpos - tr.pos0) : -1;
    if (jnew >= 0 && tid < NCH)   // the appended token's key is not in the store yet
      reinterpret_cast<int4*>(new_key)[tid] = reinterpret_cast<const int4*>(p.new_keys + (long long)tr.r * d)[tid];
    const bool ok = mbar_wait_bounded(&bar[s], (uint32_t)((k / IDX_STAGES) & 1));
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    consumed = k + 1;
    HS_TRACE_IF(p, 0, 2, tid == 0 && k == 0);
    const unsigned char* tile = stage + (size_t)s * IDX_TILE_BYTES;
    uint32_t* keys_out = p.s.scores + (long long)tr.r * p.score_stride + tr.pos0;
    for (int j = tid; j < tr.npos; j += SC_THREADS) {
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
      const uint32_t key = (uint32_t)(acc + IDX_KEY_BIAS);
      keys_out[j] = key;
      atomicAdd(&hist[key >> 12], 1u);
    }
    __syncthreads();   // stage s consumed; histogram updates of this tile done
    if (tid == 0 && k + IDX_STAGES < ntile) issue(k + IDX_STAGES);
    // end of this request's segment: add the histogram to the request's one
    int rn = r_cur;
    const bool seg_end = (k + 1 == ntile) || (prefix[rn + 1] <= t0 + k + 1);
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
      const int issued = min(ntile, consumed + IDX_STAGES);
      for (int k = consumed; k < issued; ++k)
        (void)mbar_wait_bounded(&bar[k % IDX_STAGES], (uint32_t)((k / IDX_STAGES) & 1));
      set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
    }
    __syncthreads();
  }
}

template <int NCH>
static cudaError_t run_score(const DecodeParams* p, size_t smem, cudaStream_t st) {
  auto kern = score_kernel<NCH>;
  if (p == nullptr) return allow_smem(kern, smem);
  kern<<<p->score_grid, SC_THREADS, smem, st>>>(*p);
  return cudaGetLastError();
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
