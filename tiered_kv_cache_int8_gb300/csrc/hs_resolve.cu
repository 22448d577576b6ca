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
// smallest (last-use stamp, slot), in that order; every used slot's stamp becomes
// the (request, layer) step counter, which then grows by one.
//
// Design (sm_103a), one 1024-thread CTA per request, everything in shared memory:
//  1. exact top-k over the 24-bit keys the score kernel left in L2: the first
//     digit comes from the score kernel's histogram, one pass over the keys
//     builds the second-digit histogram, and an ordered compaction (per-thread
//     contiguous ranges + block scans) emits the k positions ascending, taking
//     keys equal to the threshold in position order;
//  2. RESOLVE: hit test through the page table (independent gathers), miss
//     compaction with prefix sums, victims from an explicit LRU list — slots
//     sorted by (stamp, slot).  A call only moves the slots it used to the most
//     recent end (they all get the newest stamp, so they sort by slot among
//     themselves), so two stable compactions maintain the list: no sort, no heap;
//  3. the host fetch of the missed rows.  With fetch_mode 1 this CTA copies them
//     from the mapped pinned host copy into their slots (serial, as the pages
//     describe).  With fetch_mode 0 it marks them in slot_of_sel and the attention
//     kernel's producer copies them from host memory into its stage (and from
//     there into the slot) while the rest of the rows stream from HBM, so
//     host-link time overlaps HBM time.  Both give identical results.
#include "hs_internal.cuh"

namespace hs {

namespace {

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct ResLayout {
  size_t hist, sel, slot, miss_i, victim, used, ord, total;
};

__host__ __device__ inline ResLayout res_layout(int B, int K) {
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
  L.total = off;
  return L;
}

struct ResShared {
  int scan[2 * (RES_THREADS / 32 + 1)];
  int b1, above1, b2, above2;
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

}  // namespace

size_t resolve_smem_bytes(const Geometry& g) { return res_layout(g.hot_slots, g.top_k).total; }

__global__ void __launch_bounds__(RES_THREADS, 1) topk_resolve_kernel(DecodeParams p) {
  const Geometry& g = p.g;
  const int tid = threadIdx.x;
  const int ri = blockIdx.x;
  const int K = g.top_k;
  const int B = g.hot_slots;
  int32_t* sel_g = p.s.sel + (long long)ri * K;
  int32_t* sel_out = p.sel_out ? p.sel_out + (long long)ri * K : nullptr;
  const int req = p.req_ids ? p.req_ids[ri] : ri;
  if (req < 0 || req >= g.max_requests) {
    if (tid == 0) set_error(p.s.dev_error, HS_DEVERR_REQ_RANGE);
    if (sel_out)
      for (int i = tid; i < K; i += RES_THREADS) sel_out[i] = -1;
    return;
  }
  HS_TRACE(p, 1, 0);
  const long long rl = (long long)req * g.n_layers + p.layer;
  const int len = p.s.length[rl];

  extern __shared__ __align__(16) unsigned char smem_raw[];
  const ResLayout L = res_layout(B, K);
  __shared__ ResShared sh;
  uint32_t* h = reinterpret_cast<uint32_t*>(smem_raw + L.hist);
  int32_t* sel = reinterpret_cast<int32_t*>(smem_raw + L.sel);
  int32_t* slot_sel = reinterpret_cast<int32_t*>(smem_raw + L.slot);
  int32_t* miss_i = reinterpret_cast<int32_t*>(smem_raw + L.miss_i);
  int32_t* victim = reinterpret_cast<int32_t*>(smem_raw + L.victim);
  int32_t* ord = reinterpret_cast<int32_t*>(smem_raw + L.ord);
  uint8_t* used = smem_raw + L.used;

  // The LRU order list is needed only after the selection: start copying it
  // into shared memory now (async), so the copy overlaps the top-k passes.
  const int32_t* order_g = p.s.order + rl * B;
  for (int c4 = tid; c4 < B / 4; c4 += RES_THREADS) cp_async_16(ord + 4 * c4, order_g + 4 * c4);
  const int t_step = p.s.step[rl];

  // ---- the token appended by this call (its score was taken from the input) ----
  int N = len;
  if (p.new_kv) {
    if (len + 1 <= g.max_context) {
      N = len + 1;
      const int kvec = g.d_idx / 16;
      if (tid < kvec)
        reinterpret_cast<int4*>(p.s.idx_keys + (rl * g.max_context + len) * g.d_idx)[tid] =
            reinterpret_cast<const int4*>(p.new_keys + (long long)ri * g.d_idx)[tid];
      const int rvec = g.row_bytes / 16;
      const int4* src = reinterpret_cast<const int4*>(p.new_kv + (long long)ri * g.row_elems);
      int4* dst = reinterpret_cast<int4*>(p.s.host_kv + (rl * g.max_context + len) * g.row_elems);
      for (int v = tid; v < rvec; v += RES_THREADS) dst[v] = src[v];
      if (tid == 0) {
        p.s.length[rl] = N;
        atomicAdd(&p.s.glob[1], (unsigned long long)g.row_bytes);
      }
    } else if (tid == 0) {
      set_error(p.s.dev_error, HS_DEVERR_CAPACITY);
    }
  }
  const int kk = min(K, N);
  HS_TRACE(p, 1, 1);

  // ======================= 1. top-k, ascending =======================
  if (N <= K) {
    for (int i = tid; i < N; i += RES_THREADS) sel[i] = i;
  } else {
    const uint32_t* keys = p.s.scores + (long long)ri * p.score_stride;
    uint4* gh4 = reinterpret_cast<uint4*>(p.s.hist + (long long)ri * IDX_BINS);
    static_assert(IDX_BINS == 4 * RES_THREADS, "one 16-byte histogram chunk per thread");
    reinterpret_cast<uint4*>(h)[tid] = gh4[tid];
    gh4[tid] = make_uint4(0, 0, 0, 0);   // ready for the next call
    __syncthreads();
    select_digit(h, K, sh.scan, &sh.b1, &sh.above1);
    const int b1 = sh.b1, above1 = sh.above1;
    HS_TRACE(p, 1, 2);
    reinterpret_cast<uint4*>(h)[tid] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    // second digit: histogram of the low 12 bits of the keys inside digit b1
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
    __syncthreads();
    HS_TRACE(p, 1, 3);
    select_digit(h, K - above1, sh.scan, &sh.b2, &sh.above2);
    HS_TRACE(p, 1, 4);
    const uint32_t vstar = ((uint32_t)b1 << 12) | (uint32_t)sh.b2;
    const int need_eq = K - (above1 + sh.above2);   // >= 1
    // ordered compaction over per-thread contiguous ranges (multiples of 4 keys,
    // read as 16-byte vectors, 8 in flight; the second read hits L1)
    const int per = (((N + RES_THREADS - 1) / RES_THREADS) + 3) & ~3;
    const int j0 = min(N, tid * per), j1 = min(N, j0 + per);
    const int jv = j0 + ((j1 - j0) & ~3);
    int n_gt = 0, n_eq = 0;
    {
      int j = j0;
      for (; j + 32 <= jv; j += 32) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = *reinterpret_cast<const uint4*>(keys + j + 4 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          n_gt += (v[u].x > vstar) + (v[u].y > vstar) + (v[u].z > vstar) + (v[u].w > vstar);
          n_eq += (v[u].x == vstar) + (v[u].y == vstar) + (v[u].z == vstar) + (v[u].w == vstar);
        }
      }
      for (; j + 4 <= jv; j += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + j);
        n_gt += (v.x > vstar) + (v.y > vstar) + (v.z > vstar) + (v.w > vstar);
        n_eq += (v.x == vstar) + (v.y == vstar) + (v.z == vstar) + (v.w == vstar);
      }
      for (; j < j1; ++j) {
        const uint32_t v = keys[j];
        n_gt += v > vstar;
        n_eq += v == vstar;
      }
    }
    const int2 before = block_exclusive_scan2<RES_THREADS>(n_gt, n_eq, sh.scan, nullptr, nullptr);
    HS_TRACE(p, 1, 5);
    int o = before.x + min(before.y, need_eq);
    int eq_rank = before.y;
    auto emit = [&](int j, uint32_t v) {
      bool take = v > vstar;
      if (v == vstar) {
        take = eq_rank < need_eq;
        ++eq_rank;
      }
      if (take && o < K) sel[o++] = j;
    };
    {
      int j = j0;
      for (; j + 32 <= jv; j += 32) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = *reinterpret_cast<const uint4*>(keys + j + 4 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (max(max(v[u].x, v[u].y), max(v[u].z, v[u].w)) < vstar) continue;   // nothing taken
          emit(j + 4 * u, v[u].x);
          emit(j + 4 * u + 1, v[u].y);
          emit(j + 4 * u + 2, v[u].z);
          emit(j + 4 * u + 3, v[u].w);
        }
      }
      for (; j + 4 <= jv; j += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + j);
        emit(j, v.x);
        emit(j + 1, v.y);
        emit(j + 2, v.z);
        emit(j + 3, v.w);
      }
      for (; j < j1; ++j) emit(j, keys[j]);
    }
  }
  __syncthreads();
  HS_TRACE(p, 1, 6);
  for (int i = tid; i < K; i += RES_THREADS) {
    const int v = i < kk ? sel[i] : -1;
    if (i < kk) sel_g[i] = v;
    if (sel_out) sel_out[i] = v;
  }
  if (kk == 0) {   // nothing selected: the attention kernel writes zeros
    cp_async_wait_all();
    return;
  }

  // ======================= 2. RESOLVE metadata =======================
  int32_t* page = p.s.page + rl * g.max_context;
  int32_t* reverse = p.s.reverse + rl * B;
  int32_t* stamp = p.s.stamp + rl * B;
  int32_t* order = p.s.order + rl * B;
  const int t = t_step;
  for (int j = tid; j < B; j += RES_THREADS) used[j] = 0;
  cp_async_wait_all();   // this thread's part of the LRU list has landed
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
      }
    }
  }
  __syncthreads();   // `used` is cleared before it is marked
  for (int i = tid; i < kk; i += RES_THREADS) {
    const int sl = slot_sel[i];
    if (sl >= 0 && sl < B) used[sl] = 1;
  }
  HS_TRACE(p, 1, 7);
  if (__syncthreads_or(bad)) {
    if (tid == 0) set_error(p.s.dev_error, HS_DEVERR_METADATA);
    return;   // slot_of_sel keeps in-range values from before: the attention stays in bounds
  }
  HS_TRACE(p, 1, 8);
  // misses in ascending selection order, and the unpinned entries of the LRU list
  const int per_i = (kk + RES_THREADS - 1) / RES_THREADS;
  const int i0 = min(kk, tid * per_i), i1 = min(kk, i0 + per_i);
  const int per_j = (B + RES_THREADS - 1) / RES_THREADS;
  const int j0 = min(B, tid * per_j), j1 = min(B, j0 + per_j);
  int nm = 0, nc = 0;
  for (int i = i0; i < i1; ++i) nm += slot_sel[i] < 0;
  for (int j = j0; j < j1; ++j) nc += used[ord[j]] == 0;
  int m;
  const int2 mc = block_exclusive_scan2<RES_THREADS>(nm, nc, sh.scan, &m, nullptr);
  int mb = mc.x;
  for (int i = i0; i < i1; ++i)
    if (slot_sel[i] < 0) miss_i[mb++] = i;
  // victims: the first m unpinned entries of the LRU list
  int cb = mc.y;
  for (int j = j0; j < j1 && cb < m; ++j) {
    const int sl = ord[j];
    if (used[sl] == 0) {
      victim[cb++] = sl;
      used[sl] = 2;
    }
  }
  __syncthreads();
  HS_TRACE(p, 1, 9);
  // evict, then record the new residents
  bool incons = false;
  for (int r = tid; r < m; r += RES_THREADS) {
    const int v = victim[r];
    const int i = miss_i[r];
    const int pnew = sel[i];
    const int old = reverse[v];
    if (old >= 0) {
      if (old >= g.max_context || page[old] != v) incons = true;
      else page[old] = -1;
    }
    reverse[v] = pnew;
    page[pnew] = v;
    slot_sel[i] = v;
  }
  if (incons) set_error(p.s.dev_error, HS_DEVERR_METADATA);
  __syncthreads();
  HS_TRACE(p, 1, 10);
  // slot of every selected position (misses flagged for the attention kernel
  // when it does the fetch); stamp every used slot
  const int miss_flag = p.fetch_mode == 0 ? HS_SLOT_MISS_FLAG : 0;
  int32_t* sos = p.s.slot_of_sel + (long long)ri * K;
  for (int i = tid; i < kk; i += RES_THREADS) {
    const int sl = slot_sel[i];
    stamp[sl] = t;
    sos[i] = sl;
  }
  __syncthreads();
  for (int r = tid; r < m; r += RES_THREADS) sos[miss_i[r]] = victim[r] | miss_flag;
  HS_TRACE(p, 1, 11);
  // new LRU list: unused slots keep their order, used slots go last by slot
  int nu = 0, nus = 0;
  for (int j = j0; j < j1; ++j) nu += used[ord[j]] == 0;
  for (int sl = j0; sl < j1; ++sl) nus += used[sl] != 0;
  int n_unused;
  const int2 un = block_exclusive_scan2<RES_THREADS>(nu, nus, sh.scan, &n_unused, nullptr);
  int ub = un.x;
  for (int j = j0; j < j1; ++j) {
    const int sl = ord[j];
    if (used[sl] == 0) order[ub++] = sl;
  }
  int sb = n_unused + un.y;
  for (int sl = j0; sl < j1; ++sl)
    if (used[sl] != 0) order[sb++] = sl;
  if (tid == 0) {
    p.s.step[rl] = t + 1;
    p.s.hits[rl] += (unsigned long long)(kk - m);
    p.s.misses[rl] += (unsigned long long)m;
    atomicAdd(&p.s.glob[0], (unsigned long long)m * g.row_bytes);
  }

  HS_TRACE(p, 1, 12);
  // ======================= 3. host fetch (fetch_mode 1) =======================
  if (p.fetch_mode == 1 && m > 0) {
    const int rvec = g.row_bytes / 16;
    const long long total = (long long)m * rvec;
    const unsigned char* src_base =
        reinterpret_cast<const unsigned char*>(p.s.host_kv) + (size_t)rl * g.max_context * g.row_bytes;
    unsigned char* dst_base = reinterpret_cast<unsigned char*>(p.s.hot) + (size_t)rl * B * g.row_bytes;
    constexpr int U = 4;
    // plain (coherent) loads: the row appended above may be among the misses
    for (long long e0 = tid; e0 < total; e0 += (long long)U * RES_THREADS) {
      int4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long e = e0 + (long long)u * RES_THREADS;
        if (e < total) {
          const int q = (int)(e / rvec), cidx = (int)(e - (long long)q * rvec);
          v[u] = *reinterpret_cast<const int4*>(src_base + (size_t)sel[miss_i[q]] * g.row_bytes + cidx * 16);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long e = e0 + (long long)u * RES_THREADS;
        if (e < total) {
          const int q = (int)(e / rvec), cidx = (int)(e - (long long)q * rvec);
          *reinterpret_cast<int4*>(dst_base + (size_t)victim[q] * g.row_bytes + cidx * 16) = v[u];
        }
      }
    }
  }
  HS_TRACE(p, 1, 13);
}

cudaError_t launch_resolve(const DecodeParams& p, size_t smem, cudaStream_t st) {
  topk_resolve_kernel<<<p.n_req, RES_THREADS, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t prepare_resolve(size_t smem) {
  return allow_smem(topk_resolve_kernel, smem);
}

}  // namespace hs
