// Indexer scores + top-k selection, one thread-block cluster per request.
//
// Method: "10月14日学习笔记" (zgchen.com), "HiSparse / 动机": an indexer scores
// the context and attention runs over the top-k tokens only.  The score is an
// int8 query dotted with each position's int8 index key, summed exactly in
// int32 (dp4a); ties at the k-th score go to the lower position; the k
// positions are emitted in ascending order.
//
// Design (sm_103a):
//  * The request's positions are split over the IDX_CLUSTER CTAs of a cluster.
//    Each CTA streams its slice of index keys HBM -> shared memory with 1-D bulk
//    async copies (cp.async.bulk, mbarrier completion, IDX_STAGES deep) and
//    scores it with dp4a; the scores stay in shared memory as 24-bit keys
//    (score + 2^22), never written to HBM.
//  * Exact radix select over two 12-bit digits.  Each CTA builds a histogram of
//    its keys; the cluster reduces the histograms through distributed shared
//    memory (CTA c owns bins [c*512, c*512+512)), finds the digit holding the
//    k-th largest key, and repeats on the low digit for the keys inside it.
//  * Keys above the threshold are all taken; keys equal to it are taken in
//    position order until k is reached.  Every CTA learns the counts of the
//    CTAs before it and compacts its own slice in position order, so the output
//    is ascending without a sort.
#include <cooperative_groups.h>

#include "hs_internal.cuh"

namespace cg = cooperative_groups;

namespace hs {

namespace {

struct IdxShared {
  uint64_t bar[IDX_STAGES];
  int scan[IDX_THREADS / 32 + 1];
  int seg_tot[IDX_CLUSTER];
  int cnt_gt[IDX_CLUSTER];
  int cnt_eq[IDX_CLUSTER];
  int bstar;       // selected digit of the current level
  int above;       // keys above that digit (whole request)
  int flag;
};

constexpr int SEG = IDX_BINS / IDX_CLUSTER;   // histogram bins owned by one CTA

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

size_t indexer_smem_bytes(const Geometry& g, int chunk_max) {
  (void)g;
  size_t off = align_up(sizeof(IdxShared), 128);
  off += IDX_BINS * sizeof(uint32_t);           // histogram
  off += SEG * sizeof(int);                     // reduced own segment
  off = align_up(off, 128);
  off += (size_t)IDX_STAGES * IDX_TILE_BYTES;   // key staging
  off += (size_t)chunk_max * sizeof(uint32_t);  // scores of this CTA's slice
  return off;
}

// One level of the cluster-wide radix select.  On entry every CTA's `hist`
// holds its local histogram; `kneed` is how many keys are still needed from the
// top of the candidate set.  On exit sh.bstar / sh.above are set in every CTA.
__device__ __forceinline__ void cluster_select_digit(cg::cluster_group& cluster, IdxShared& sh,
                                                     uint32_t* hist, int* seg, int kneed) {
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  cluster.sync();  // every local histogram is complete
  for (int b = tid; b < SEG; b += IDX_THREADS) {
    int acc = 0;
#pragma unroll
    for (int c = 0; c < IDX_CLUSTER; ++c) {
      const uint32_t* rh = cluster.map_shared_rank(hist, c);
      acc += (int)rh[rank * SEG + b];
    }
    seg[b] = acc;
  }
  __syncthreads();
  int local = 0;
  for (int b = tid; b < SEG; b += IDX_THREADS) local += seg[b];
  const int tot = block_sum<IDX_THREADS>(local, sh.scan);
  if (tid < IDX_CLUSTER) {
    IdxShared* rs = cluster.map_shared_rank(&sh, tid);
    rs->seg_tot[rank] = tot;
  }
  cluster.sync();  // segment totals visible everywhere; remote histogram reads done
  int above = 0;
  for (int c = rank + 1; c < IDX_CLUSTER; ++c) above += sh.seg_tot[c];
  if (above < kneed && kneed <= above + sh.seg_tot[rank]) {
    // the k-th largest key falls in this CTA's bins: scan them from the top
    static_assert(SEG <= IDX_THREADS, "one bin per thread");
    const int b = SEG - 1 - tid;
    const int v = (tid < SEG) ? seg[b] : 0;
    int tot2;
    const int excl = block_exclusive_scan<IDX_THREADS>(v, sh.scan, &tot2);
    if (tid < SEG && above + excl < kneed && kneed <= above + excl + v) {
      const int bstar = rank * SEG + b;
      const int ab = above + excl;
      for (int c = 0; c < IDX_CLUSTER; ++c) {
        IdxShared* rs = cluster.map_shared_rank(&sh, c);
        rs->bstar = bstar;
        rs->above = ab;
      }
    }
  }
  cluster.sync();  // the selected digit is visible everywhere
}

__global__ void __launch_bounds__(IDX_THREADS, 1) indexer_topk_kernel(DecodeParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  const Geometry& g = p.g;
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int ri = blockIdx.y;
  const int req = p.req_ids ? p.req_ids[ri] : ri;
  const int K = g.top_k;
  int32_t* sel = p.s.sel + (long long)ri * K;
  int32_t* sel_out = p.sel_out ? p.sel_out + (long long)ri * K : nullptr;

  if (req < 0 || req >= g.max_requests) {   // uniform over the cluster
    if (rank == 0 && tid == 0) set_error(p.s.dev_error, HS_DEVERR_REQ_RANGE);
    if (rank == 0)
      for (int i = tid; i < K; i += IDX_THREADS) {
        sel[i] = -1;
        if (sel_out) sel_out[i] = -1;
      }
    return;
  }
  const long long rl = (long long)req * g.n_layers + p.layer;
  const int N = p.s.length[rl];
  if (N <= K) {   // every position is selected (or none): no scoring needed
    if (rank == 0)
      for (int i = tid; i < K; i += IDX_THREADS) {
        const int v = i < N ? i : -1;
        sel[i] = v;
        if (sel_out) sel_out[i] = v;
      }
    return;
  }

  extern __shared__ __align__(128) unsigned char smem_raw[];
  IdxShared& sh = *reinterpret_cast<IdxShared*>(smem_raw);
  size_t off = align_up(sizeof(IdxShared), 128);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw + off);
  off += IDX_BINS * sizeof(uint32_t);
  int* seg = reinterpret_cast<int*>(smem_raw + off);
  off += SEG * sizeof(int);
  off = align_up(off, 128);
  unsigned char* stage = smem_raw + off;
  off += (size_t)IDX_STAGES * IDX_TILE_BYTES;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + off);

  const int d = g.d_idx;
  int chunk = (N + IDX_CLUSTER - 1) / IDX_CLUSTER;
  chunk = (chunk + 31) & ~31;
  const int start = min(N, rank * chunk);
  const int count = min(N, start + chunk) - start;

  for (int b = tid; b < IDX_BINS; b += IDX_THREADS) hist[b] = 0;
  if (tid == 0) {
    for (int s = 0; s < IDX_STAGES; ++s) mbar_init(&sh.bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- scores: stream the slice's index keys through shared memory ------------
  const int TP = IDX_TILE_BYTES / d;   // positions per tile
  const int n_tiles = (count + TP - 1) / TP;
  const int8_t* gkeys = p.s.idx_keys + (rl * g.max_context + start) * d;
  auto issue = [&](int i) {
    const int s = i % IDX_STAGES;
    const int npos = min(TP, count - i * TP);
    const uint32_t bytes = (uint32_t)(npos * d);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&sh.bar[s], bytes);
    bulk_g2s(stage + (size_t)s * IDX_TILE_BYTES, gkeys + (size_t)i * TP * d, bytes, &sh.bar[s]);
  };
  if (tid == 0)
    for (int i = 0; i < IDX_STAGES && i < n_tiles; ++i) issue(i);

  const int lpp = d >> 4;              // lanes per position (16 bytes each)
  const int sub = tid & (lpp - 1);
  const int pl = tid / lpp;
  const int ppp = IDX_THREADS / lpp;   // positions per pass
  const int4 qv = *reinterpret_cast<const int4*>(p.q_idx + (long long)ri * d + sub * 16);

  bool timed_out = false;
  int consumed = 0;
  for (int i = 0; i < n_tiles; ++i) {
    const int s = i % IDX_STAGES;
    const bool ok = mbar_wait_bounded(&sh.bar[s], (uint32_t)((i / IDX_STAGES) & 1));
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    consumed = i + 1;
    const unsigned char* tile = stage + (size_t)s * IDX_TILE_BYTES;
    const int npos = min(TP, count - i * TP);
    for (int b = 0; b < npos; b += ppp) {
      const int j = b + pl;
      int acc = 0;
      if (j < npos) {
        const int4 kv = *reinterpret_cast<const int4*>(tile + j * d + sub * 16);
        acc = __dp4a(kv.x, qv.x, acc);
        acc = __dp4a(kv.y, qv.y, acc);
        acc = __dp4a(kv.z, qv.z, acc);
        acc = __dp4a(kv.w, qv.w, acc);
      }
      for (int o = lpp >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, o);
      if (sub == 0 && j < npos) {
        const uint32_t key = (uint32_t)(acc + IDX_KEY_BIAS);
        keys[i * TP + j] = key;
        atomicAdd(&hist[key >> 12], 1u);
      }
    }
    __syncthreads();
    if (tid == 0 && i + IDX_STAGES < n_tiles) issue(i + IDX_STAGES);
  }
  if (timed_out) {
    // drain copies still in flight (bounded) before the buffers go away
    if (tid == 0) {
      const int issued = min(n_tiles, consumed + IDX_STAGES);
      for (int i = consumed; i < issued; ++i)
        (void)mbar_wait_bounded(&sh.bar[i % IDX_STAGES], (uint32_t)((i / IDX_STAGES) & 1));
      set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
    }
    __syncthreads();
  }

  // ---- level 1: high 12 bits --------------------------------------------------
  cluster_select_digit(cluster, sh, hist, seg, K);
  const int b1 = sh.bstar;
  const int above1 = sh.above;
  // ---- level 2: low 12 bits of the keys inside digit b1 -----------------------
  for (int b = tid; b < IDX_BINS; b += IDX_THREADS) hist[b] = 0;
  __syncthreads();
  for (int j = tid; j < count; j += IDX_THREADS) {
    const uint32_t key = keys[j];
    if ((int)(key >> 12) == b1) atomicAdd(&hist[key & 4095u], 1u);
  }
  __syncthreads();
  cluster_select_digit(cluster, sh, hist, seg, K - above1);
  const uint32_t vstar = ((uint32_t)b1 << 12) | (uint32_t)sh.bstar;
  const int cnt_gt_all = above1 + sh.above;
  const int need_eq = K - cnt_gt_all;   // >= 1

  // ---- ordered compaction -----------------------------------------------------
  const int per = (count + IDX_THREADS - 1) / IDX_THREADS;
  const int j0 = min(count, tid * per);
  const int j1 = min(count, j0 + per);
  int n_gt = 0, n_eq = 0;
  for (int j = j0; j < j1; ++j) {
    const uint32_t key = keys[j];
    n_gt += key > vstar;
    n_eq += key == vstar;
  }
  int tot_gt, tot_eq;
  const int eq_before_t = block_exclusive_scan<IDX_THREADS>(n_eq, sh.scan, &tot_eq);
  (void)block_exclusive_scan<IDX_THREADS>(n_gt, sh.scan, &tot_gt);
  if (tid < IDX_CLUSTER) {
    IdxShared* rs = cluster.map_shared_rank(&sh, tid);
    rs->cnt_gt[rank] = tot_gt;
    rs->cnt_eq[rank] = tot_eq;
  }
  cluster.sync();
  int out_base = 0, eq_seen = 0, my_take_eq = 0;
  for (int c = 0; c < IDX_CLUSTER; ++c) {
    const int take = max(0, min(need_eq - eq_seen, sh.cnt_eq[c]));
    if (c < rank) out_base += sh.cnt_gt[c] + take;
    if (c == rank) my_take_eq = take;
    eq_seen += sh.cnt_eq[c];
  }
  const int my_eq_take_t = max(0, min(my_take_eq - eq_before_t, n_eq));
  const int n_sel_t = n_gt + my_eq_take_t;
  int o = out_base + block_exclusive_scan<IDX_THREADS>(n_sel_t, sh.scan, nullptr);
  int eq_rank = eq_before_t;
  for (int j = j0; j < j1; ++j) {
    const uint32_t key = keys[j];
    bool take = key > vstar;
    if (key == vstar) {
      take = eq_rank < my_take_eq;
      ++eq_rank;
    }
    if (take) {
      const int pos = start + j;
      if (o < K) {
        sel[o] = pos;
        if (sel_out) sel_out[o] = pos;
      }
      ++o;
    }
  }
  cluster.sync();   // keep this CTA's shared memory alive until remote readers are done
}

cudaError_t launch_indexer_topk(const DecodeParams& p, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(IDX_CLUSTER, p.n_req, 1);
  lc.blockDim = dim3(IDX_THREADS, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = IDX_CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, indexer_topk_kernel, p);
}

cudaError_t prepare_indexer(size_t smem) {
  return cudaFuncSetAttribute(indexer_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace hs
