// RESOLVE: hit test, LRU replacement, metadata update and host fetch of the
// missed rows, fused in one launch per layer (one thread-block cluster per
// request).
//
// Method: "KV卸载上主机:HiSparse、PDD与DDR4回收", section "论文1：HiSparse" —
// a page table plus LRU metadata drive replacement of the B hot slots of each
// (request, layer), and hit detection, LRU replacement, metadata update and the
// host fetch are fused into one RESOLVE kernel per layer.  "10月14日学习笔记",
// "HiSparse / 方法" item 1: LRU replacement.
//
// Replacement rule: slots holding a selected position (hits) are pinned; the
// m misses, taken in ascending position order, go to the m unpinned slots with
// the smallest (last-use stamp, slot), in that order; every used slot's stamp
// becomes the (request, layer) step counter, which then grows by one.
//
// Design (sm_103a): the LRU order is kept explicitly as a list of slots sorted
// by (stamp, slot).  A call only ever moves the slots it used to the most
// recent end (they all get the newest stamp, so among themselves they sort by
// slot), so the list is maintained by two stable block-wide compactions per
// call and the victims are simply the first m unpinned entries: no sort and no
// heap.  The cluster's rank-0 CTA does the metadata work in shared memory and
// publishes the (position, slot) list of the misses; all CTAs of the cluster
// then pull their share of the missed rows from the mapped pinned host copy
// with 16-byte loads (several in flight per thread) straight into the slots.
#include <cooperative_groups.h>

#include "hs_internal.cuh"

namespace cg = cooperative_groups;

namespace hs {

namespace {

struct ResShared {
  int scan[RES_THREADS / 32 + 1];
  int m;          // misses of this call (published by rank 0)
  int abort;      // rank 0 found an inconsistency: nothing to copy
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct ResLayout {
  size_t used, ord, a, b, c, d, total;
};

__host__ __device__ inline ResLayout res_layout(int B, int K) {
  ResLayout L;
  size_t off = (sizeof(ResShared) + 15) / 16 * 16;
  L.used = off;
  off += (size_t)(B + 15) / 16 * 16;   // uint8 flags: 0 free, 1 hit, 2 victim
  L.ord = off;
  off += (size_t)B * 4;
  L.a = off;                           // slot of each selected position (rank 0) / my positions
  off += (size_t)K * 4;
  L.b = off;                           // selection index of each miss (rank 0) / my slots
  off += (size_t)K * 4;
  L.c = off;                           // position of each miss
  off += (size_t)K * 4;
  L.d = off;                           // victim slot of each miss
  off += (size_t)K * 4;
  L.total = off;
  return L;
}

}  // namespace

size_t resolve_smem_bytes(const Geometry& g) { return res_layout(g.hot_slots, g.top_k).total; }

__global__ void __launch_bounds__(RES_THREADS, 1) resolve_kernel(DecodeParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  const Geometry& g = p.g;
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int ri = blockIdx.y;
  const int req = p.req_ids ? p.req_ids[ri] : ri;
  if (req < 0 || req >= g.max_requests) return;   // reported by the indexer kernel
  const long long rl = (long long)req * g.n_layers + p.layer;
  const int N = p.s.length[rl];
  const int K = g.top_k;
  const int B = g.hot_slots;
  const int kk = min(K, N);
  if (kk == 0) return;   // uniform over the cluster

  extern __shared__ __align__(16) unsigned char smem_raw[];
  const ResLayout L = res_layout(B, K);
  ResShared& sh = *reinterpret_cast<ResShared*>(smem_raw);
  uint8_t* used = smem_raw + L.used;
  int32_t* ord = reinterpret_cast<int32_t*>(smem_raw + L.ord);
  int32_t* a_arr = reinterpret_cast<int32_t*>(smem_raw + L.a);
  int32_t* b_arr = reinterpret_cast<int32_t*>(smem_raw + L.b);
  int32_t* miss_pos = reinterpret_cast<int32_t*>(smem_raw + L.c);
  int32_t* victim = reinterpret_cast<int32_t*>(smem_raw + L.d);

  if (rank == 0) {
    const int32_t* sel = p.s.sel + (long long)ri * K;
    int32_t* slot_of_sel = p.s.slot_of_sel + (long long)ri * K;
    int32_t* page = p.s.page + rl * g.max_context;
    int32_t* reverse = p.s.reverse + rl * B;
    int32_t* stamp = p.s.stamp + rl * B;
    int32_t* order = p.s.order + rl * B;
    const int t = p.s.step[rl];
    int32_t* slot_sel = a_arr;   // slot of each selected position, -1 = miss
    int32_t* miss_i = b_arr;

    for (int j = tid; j < B; j += RES_THREADS) {
      used[j] = 0;
      ord[j] = order[j];
    }
    __syncthreads();

    // 1. hit test through the page table; pin hit slots
    const int per_i = (kk + RES_THREADS - 1) / RES_THREADS;
    const int i0 = min(kk, tid * per_i), i1 = min(kk, i0 + per_i);
    int nm = 0;
    bool bad = false;
    for (int i = i0; i < i1; ++i) {
      const int pos = sel[i];
      int s = -1;
      if (pos < 0 || pos >= N) {
        bad = true;
      } else {
        s = page[pos];
        if (s >= B) bad = true;
      }
      slot_sel[i] = s;
      if (s >= 0 && s < B) used[s] = 1;
      else ++nm;
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) {
        set_error(p.s.dev_error, HS_DEVERR_METADATA);
        sh.m = 0;
        sh.abort = 1;
      }
    } else {
      // 2. misses in ascending position (= selection) order
      int m;
      int mb = block_exclusive_scan<RES_THREADS>(nm, sh.scan, &m);
      for (int i = i0; i < i1; ++i)
        if (slot_sel[i] < 0) {
          miss_i[mb] = i;
          miss_pos[mb] = sel[i];
          ++mb;
        }
      // 3. victims: the first m unpinned entries of the LRU list
      const int per_j = (B + RES_THREADS - 1) / RES_THREADS;
      const int j0 = min(B, tid * per_j), j1 = min(B, j0 + per_j);
      int nc = 0;
      for (int j = j0; j < j1; ++j) nc += used[ord[j]] == 0;
      int cb = block_exclusive_scan<RES_THREADS>(nc, sh.scan, nullptr);
      for (int j = j0; j < j1 && cb < m; ++j) {
        const int s = ord[j];
        if (used[s] == 0) {
          victim[cb] = s;
          used[s] = 2;
          ++cb;
        }
      }
      __syncthreads();
      // 4. evict, then record the new residents
      bool incons = false;
      for (int r = tid; r < m; r += RES_THREADS) {
        const int v = victim[r];
        const int pnew = miss_pos[r];
        const int old = reverse[v];
        if (old >= 0) {
          if (old >= g.max_context || page[old] != v) incons = true;
          else page[old] = -1;
        }
        reverse[v] = pnew;
        page[pnew] = v;
        slot_sel[miss_i[r]] = v;
      }
      if (incons) set_error(p.s.dev_error, HS_DEVERR_METADATA);
      __syncthreads();
      // 5. slot of every selected position; stamp every used slot
      for (int i = tid; i < kk; i += RES_THREADS) {
        const int s = slot_sel[i];
        slot_of_sel[i] = s;
        stamp[s] = t;
      }
      // 6. new LRU list: unused slots keep their order, used slots go last by slot
      int n_unused;
      int nu = 0;
      for (int j = j0; j < j1; ++j) nu += used[ord[j]] == 0;
      int ub = block_exclusive_scan<RES_THREADS>(nu, sh.scan, &n_unused);
      for (int j = j0; j < j1; ++j) {
        const int s = ord[j];
        if (used[s] == 0) order[ub++] = s;
      }
      int nus = 0;
      for (int s = j0; s < j1; ++s) nus += used[s] != 0;
      int sb = n_unused + block_exclusive_scan<RES_THREADS>(nus, sh.scan, nullptr);
      for (int s = j0; s < j1; ++s)
        if (used[s] != 0) order[sb++] = s;
      if (tid == 0) {
        p.s.step[rl] = t + 1;
        p.s.hits[rl] += (unsigned long long)(kk - m);
        p.s.misses[rl] += (unsigned long long)m;
        atomicAdd(&p.s.glob[0], (unsigned long long)m * g.row_bytes);
        sh.m = m;
        sh.abort = 0;
      }
    }
  }
  cluster.sync();   // rank 0's miss list is complete

  // ---- pull the missed rows: host copy -> hot slots, split over the cluster ------
  ResShared* lead = cluster.map_shared_rank(&sh, 0);
  const int m = lead->m;
  const int32_t* lead_pos = cluster.map_shared_rank(miss_pos, 0);
  const int32_t* lead_vic = cluster.map_shared_rank(victim, 0);
  int32_t* my_pos = a_arr;
  int32_t* my_slot = b_arr;
  const int n_my = m > rank ? (m - rank + RES_CLUSTER - 1) / RES_CLUSTER : 0;
  for (int q = tid; q < n_my; q += RES_THREADS) {
    my_pos[q] = lead_pos[rank + q * RES_CLUSTER];
    my_slot[q] = lead_vic[rank + q * RES_CLUSTER];
  }
  __syncthreads();
  cluster.sync();   // remote reads of rank 0's shared memory are finished

  const int rvec = g.row_bytes / 16;
  const long long total = (long long)n_my * rvec;
  const unsigned char* src_base = reinterpret_cast<const unsigned char*>(p.s.host_kv) +
                                  (size_t)rl * g.max_context * g.row_bytes;
  unsigned char* dst_base = reinterpret_cast<unsigned char*>(p.s.hot) + (size_t)rl * B * g.row_bytes;
  constexpr int U = 4;
  for (long long e0 = tid; e0 < total; e0 += (long long)U * RES_THREADS) {
    int4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long e = e0 + (long long)u * RES_THREADS;
      if (e < total) {
        const int q = (int)(e / rvec), c = (int)(e - (long long)q * rvec);
        v[u] = ld_nc_v4(src_base + (size_t)my_pos[q] * g.row_bytes + c * 16);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long e = e0 + (long long)u * RES_THREADS;
      if (e < total) {
        const int q = (int)(e / rvec), c = (int)(e - (long long)q * rvec);
        *reinterpret_cast<int4*>(dst_base + (size_t)my_slot[q] * g.row_bytes + c * 16) = v[u];
      }
    }
  }
}

cudaError_t launch_resolve(const DecodeParams& p, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(RES_CLUSTER, p.n_req, 1);
  lc.blockDim = dim3(RES_THREADS, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = RES_CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, resolve_kernel, p);
}

cudaError_t prepare_resolve(size_t smem) {
  return cudaFuncSetAttribute(resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace hs
