// Sparse attention over the selected rows (GQA, head dim 128), fused with the
// host fetch of the missed rows RESOLVE left to it and with the merge of its
// partials: a persistent, warp-specialised flash-decode kernel that works
// through a queue of chunks while the select kernel is still resolving later
// requests.  The merge kernel further down serves latent rows.
//
// Method: "Heterogeneous LLM Serving with General-Purpose Processing-Near-Memory
// for Retrieval-Based Sparse Attention" (vsvnakers.github.io), "核心公式与算法",
// formula 2: softmax(Q K^T / sqrt(d_k), masked to the retrieved entries) V —
// read as a softmax over the selected positions only.  "KV卸载上主机:
// HiSparse、PDD与DDR4回收", "论文1：HiSparse": the attention math is unchanged
// by the cache, so the result must not depend on where the rows sit; missed rows
// come from the authoritative copy in pinned host memory.
//
// Design (sm_103a).  HBM-bound (each K/V byte is used by the h_q / h_kv query
// heads of its group only):
//  * Persistent grid, one CTA per SM, launched as a programmatic dependent of
//    the select kernel and started on the SMs its scorers free.  The work is a
//    queue of chunks (64 selected rows of one request, in selection order),
//    request after request, taken with a global atomic counter.  A chunk waits
//    (bounded) for its request's ready flag; requests are published in about
//    queue order, so a CTA rarely waits.
//  * Warp 8 (loader) reads the slots of a whole chunk at once (those of the next
//    chunk already while it streams this one, when that request is published),
//    then per unit
//    (16 rows per warp slice) copies every hit row (all kv heads: one
//    contiguous hot slot) HBM -> shared memory with one 1-D bulk async copy into
//    a row-padded layout (16 extra bytes per row put the 8 rows of an ldmatrix
//    phase in 8 bank groups).  Warp 9 (fetcher) copies the unit's missed rows
//    from the mapped pinned host copy with 16-byte cp.async, so slow host reads
//    never hold up the loader's own loads.  Up to 3 stages, full/empty
//    mbarriers, a descriptor per stage.
//  * Warp 10 (prefetcher) claims requests in order (a global counter) and, as
//    soon as RESOLVE has listed a request's misses (before it publishes the
//    request), starts every missed row moving over the host link into L2 (one
//    bulk prefetch per row): the link is the scarce resource, so its reads start
//    as early as the misses are known, and the fetchers later read L2.  (A bulk prefetch of host memory can hold its issuing thread for
//    microseconds, so it runs on a warp of its own.)
//  * Warps 0-7 consume: warp w serves kv head w % h_kv and row slice w / h_kv.
//    S^T = K Q^T and O^T += V^T P^T run on mma.sync m16n8k16 (bf16 in, fp32
//    accumulate) with the unit's 16 rows as M and the group's query heads as N
//    (8 per n-tile); K and V fragments come from shared memory with ldmatrix
//    (.trans for V), P^T moves into the A layout by movmatrix.  Online softmax
//    per head in fp32 (exp2, scale * log2(e) applied to the fp32 scores); P
//    enters the second product as bf16.  Once a unit has landed, the fetcher writes the
//    rows it fetched into their hot slots (bulk shared -> global copy), so later
//    steps hit; a stage is released by the 8 consumers and the fetcher.
//  * Each (chunk, slice) writes a partial (m, l, o) and counts its chunk done
//    (release).  A CTA out of chunks merges: items (request, 8 heads) in request
//    order, each once its request's chunks are all counted; per head one warp
//    finds the weights, then each thread sums one float4 of a head's output over
//    the partials in chunk order.  Rows are visited in ascending selection order
//    and chunks depend only on k_eff, so the output is bit-identical for any B and
//    any schedule.  (Latent rows use the separate merge kernel further down.)
//  * Counters of the call reset themselves: the last CTA to leave clears the
//    queues, the ready flags and the chunk counters.  Each CTA waits for the
//    select kernel to complete before it exits, so the next launch on the stream
//    sees both kernels finished.
#include <cuda_bf16.h>

#include "hs_internal.cuh"

namespace hs {

namespace {

constexpr int D = 128;
constexpr int NCONS = 8;                   // consumer warps
constexpr int LOADER = NCONS;              // warp index of the loader
constexpr int FETCHER = NCONS + 1;         // warp index of the host fetcher
constexpr int PREFETCHER = NCONS + 2;      // warp index of the host-row prefetcher
constexpr int THREADS = (NCONS + 3) * 32;
constexpr int MAX_STAGES = 3;
constexpr int TILE_MAX = 128;   // rows of a unit at h_kv = 1 (8 slices of 16)
constexpr int CHUNK_ROWS_MIN = 64;
constexpr int BAR_VOTE = 2;     // named barrier: the consumers' vote on a failed wait
constexpr int BAR_CHUNK = 3;    // named barrier: the consumers at the end of a chunk
constexpr int MERGE_HEADS = 8;  // heads per merge item (32 threads per head of 128 dims)

enum { DESC_UNIT = 0, DESC_STOP = 2 };
struct __align__(16) Desc {
  int type, ri, c, row0, nr, first, last, nmiss;   // nmiss: rows of the unit the fetcher copies
  int nxt, pad0, pad1, pad2;                       // nxt: the next chunk's request (last unit), or -1
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline int att_tile(const Geometry& g) { return ATT_SUBTILE * (NCONS / g.h_kv); }
__host__ __device__ inline int att_chunk_rows(const Geometry& g) {
  const int t = att_tile(g);
  return t >= CHUNK_ROWS_MIN ? t : (CHUNK_ROWS_MIN / t) * t;
}
__host__ __device__ inline int att_nchunk(const Geometry& g) {
  return (g.top_k + att_chunk_rows(g) - 1) / att_chunk_rows(g);
}

struct AttLayout {
  size_t bar, desc, slot_tab, mpos, stage, stage_bytes, total;
};

// Shared memory: barriers | per-stage descriptors | per-stage hot slots and host
// positions of fetched rows | stages.
__host__ __device__ inline AttLayout att_layout(const Geometry& g, int nstage) {
  AttLayout L;
  const int tile = att_tile(g);
  const size_t row_stride = (size_t)g.row_bytes + ATT_ROW_PAD;
  size_t off = 0;
  L.bar = off;
  off += 8 * (3 * MAX_STAGES) + 16;   // full/empty/descriptor barriers, flags
  off = align_up(off, 128);
  L.desc = off;
  off += sizeof(Desc) * MAX_STAGES;
  L.slot_tab = off;
  off += (size_t)MAX_STAGES * TILE_MAX * 4;   // hot slot of each fetched row (-1: none)
  L.mpos = off;
  off += (size_t)MAX_STAGES * TILE_MAX * 4;   // host position of each fetched row (-1: none)
  off = align_up(off, 128);
  L.stage = off;
  L.stage_bytes = align_up((size_t)tile * row_stride, 128);
  off += (size_t)nstage * L.stage_bytes;
  L.total = align_up(off, 128);
  return L;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// The transpose of an 8x8 b16 matrix held in the mma fragment layout (lane l:
// row l / 4, columns 2 (l % 4) and +1), returned in the same layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// The mbarrier receives one arrival once all of this thread's earlier cp.async
// copies have landed (its pending count is raised first, so the phase cannot
// complete before then).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bulk copy shared -> global (hot slot), tracked per thread by bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Bounded wait that also gives up once another warp has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* err, unsigned long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit) {
        *abort_flag = 1;
        set_error(err, HS_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

}  // namespace

int attention_parts(const Geometry& g) {
  if (g.shared_kv) return mla_parts(g);
  return att_nchunk(g) * (NCONS / g.h_kv);
}

// Three stages where they fit, else two.
static int attention_stages(const Geometry& g, size_t limit) {
  return att_layout(g, MAX_STAGES).total <= limit ? MAX_STAGES : 2;
}

size_t attention_smem_bytes(const Geometry& g) {
  if (g.shared_kv) return mla_smem_bytes(g);
  return att_layout(g, attention_stages(g, 227 * 1024)).total;
}

template <int G, int HKV>
__global__ void __launch_bounds__(THREADS, 1) attn_gqa_kernel(DecodeParams p, int nstage) {
  constexpr int NSLICE = NCONS / HKV;
  constexpr int TILE = ATT_SUBTILE * NSLICE;
  constexpr int HQ = HKV * G;
  constexpr int CR = TILE >= CHUNK_ROWS_MIN ? TILE : (CHUNK_ROWS_MIN / TILE) * TILE;   // rows per chunk
  constexpr int NJC = CR / 32;                                                          // rows per lane per chunk
  constexpr int NJU = (TILE + 31) / 32;                                                 // rows per lane per unit
  const Geometry& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = g.top_k;
  const int NCHK = (K + CR - 1) / CR;
  const int NPARTS = NCHK * NSLICE;
  const long long total = (long long)p.n_req * NCHK;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  const AttLayout L = att_layout(g, nstage);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + L.bar);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* dready = empty + MAX_STAGES;   // the loader's descriptor of a stage is written
  volatile int* abort_flag = reinterpret_cast<volatile int*>(dready + MAX_STAGES);
  Desc* desc = reinterpret_cast<Desc*>(smem_raw + L.desc);
  int* slot_tab = reinterpret_cast<int*>(smem_raw + L.slot_tab);   // [stage][TILE]: hot slot of a fetched row
  int* mpos = reinterpret_cast<int*>(smem_raw + L.mpos);           // [stage][TILE]: its host position
  unsigned char* stage = smem_raw + L.stage;
  const int row_stride = g.row_bytes + ATT_ROW_PAD;
  const int rvec = g.row_bytes / 16;
  HS_TRACE(p, 2, 0);
  // this CTA's timeline and its consumers' stage waits (hs_stats): thread 0,
  // a consumer, times them
  __shared__ unsigned long long s_wait[5];   // host ns, host stages, hbm ns, hbm stages, CTA start

  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(&full[s], 2);      // the loader's arrival (with the hit bytes) and the fetcher's
      mbar_init(&empty[s], NCONS + 1);   // the consumers and the fetcher
      mbar_init(&dready[s], 1);
    }
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) s_wait[i] = 0;
    s_wait[4] = global_timer_ns();
    fence_mbar_init();
  }
  // no griddepcontrol.wait here: everything the select kernel writes for a
  // request is published through that request's ready flag
  griddep_launch_dependents();
  __syncthreads();
  HS_TRACE(p, 2, 1);

  if (warp == LOADER) {
    // ============================ loader warp ============================
    const uint64_t stream_policy = l2_evict_first_policy();   // hit rows are read once per call
    int s = 0;
    long long it = 0;
    bool dead = false;
    unsigned long long tw_ready = 0, tw_empty = 0;   // summed waits (trace builds only)
    int n_items = 0;
    auto take_stage = [&]() -> bool {   // wait until stage s may be refilled
      if (it < nstage) return true;
      const unsigned long long t0 = HS_TNOW();
      const bool ok = __all_sync(FULL_MASK, wait_or_abort(&empty[s], (uint32_t)(((it / nstage) + 1) & 1), abort_flag,
                                                          p.s.dev_error, 4 * WAIT_LIMIT_NS));
      tw_empty += HS_TNOW() - t0;
      return ok;
    };
    // a chunk's metadata: k_eff (the request's ready flag holds k_eff + 1), the
    // request id, the slots and positions of its rows (one batch of loads)
    struct Meta {
      int kk, req;
      int slot[NJC], pos[NJC];
    };
    auto load_rows = [&](Meta& m, int r, int c) {
      const int row0 = c * CR;
      const int nrows = max(0, min(CR, m.kk - row0));
      const int32_t* sos = p.s.slot_of_sel + (long long)r * K + row0;
      const int32_t* selr = p.s.sel + (long long)r * K + row0;
#pragma unroll
      for (int j = 0; j < NJC; ++j) {
        const int i = lane + 32 * j;
        m.slot[j] = i < nrows ? __ldcg(sos + i) : 0;
        m.pos[j] = i < nrows ? __ldcg(selr + i) : 0;
      }
      m.req = p.req_ids ? p.req_ids[r] : r;
    };
    unsigned nxt = 0;   // lane 0: the queue index after the current one
    if (lane == 0) nxt = atomicAdd(&p.s.sync[2], 1u);
    long long cur = (long long)__shfl_sync(FULL_MASK, nxt, 0);
    if (lane == 0 && cur < total) nxt = atomicAdd(&p.s.sync[2], 1u);
    Meta pf;                // metadata of the next chunk, when it was ready early
    long long pf_item = -1;
    bool pf_warm = false;   // its hit rows were sent towards L2
    while (!dead && cur < total) {
      const long long item = cur;
      const int r = (int)(item / NCHK);
      const int c = (int)(item % NCHK);
      Meta mt;
      if (pf_item == item) {
        mt = pf;
      } else {   // wait for the request's publication
        unsigned v = 0;
        const unsigned long long t0 = HS_TNOW();
        if (lane == 0) {
          v = wait_counter(p.s.ready + r, 1u) ? ld_acquire(p.s.ready + r) : 0u;
          if (v == 0u) set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
        }
        tw_ready += HS_TNOW() - t0;
        v = __shfl_sync(FULL_MASK, v, 0);
        mt.kk = v ? (int)v - 1 : 0;
        load_rows(mt, r, c);
      }
      const int kk = mt.kk;
      const int req = mt.req;
      const int row0 = c * CR;
      const int nrows = max(0, min(CR, kk - row0));
      if (c == 0 && lane == 0) p.s.att_nparts[r] = ((kk + CR - 1) / CR) * NSLICE;   // for the merge kernel
      int cslot[NJC], cpos[NJC];
#pragma unroll
      for (int j = 0; j < NJC; ++j) {
        cslot[j] = mt.slot[j];
        cpos[j] = mt.pos[j];
      }
      const long long rl = (long long)req * g.n_layers + p.layer;
      const unsigned char* hot =
          reinterpret_cast<const unsigned char*>(p.s.hot) + (size_t)rl * g.hot_slots * g.row_bytes;
      // a chunk past k_eff still goes through the consumers (it counts as done)
      const int nunits = nrows > 0 ? (nrows + TILE - 1) / TILE : 1;
      for (int u = 0; u < nunits; ++u) {
        const int ur0 = u * TILE;   // first row of the unit within the chunk
        const int unr = max(0, min(TILE, nrows - ur0));
        if (!take_stage()) {
          dead = true;
          break;
        }
        unsigned char* st_s = stage + (size_t)s * L.stage_bytes;
        int* tab = slot_tab + s * TILE_MAX;
        int* mp = mpos + s * TILE_MAX;
        // rows past the end of the chunk: zero them so their masked (weight-0)
        // values stay finite
        if (unr < TILE) {
          for (int e = lane; e < (TILE - unr) * rvec; e += 32) {
            const int i = unr + e / rvec;
            *reinterpret_cast<int4*>(st_s + (size_t)i * row_stride + (e % rvec) * 16) = make_int4(0, 0, 0, 0);
          }
        }
        // the unit's rows: lane l takes rows l, l + 32, ... of the unit; row i of
        // the unit is row ur0 + i of the chunk, held by lane (ur0 + i) % 32 in
        // word (ur0 + i) / 32 of the chunk's batch (every lane joins every shuffle)
        int usl[NJU];
        int hit_rows = 0, miss_rows = 0;
#pragma unroll
        for (int m = 0; m < NJU; ++m) {
          const int i = lane + 32 * m;
          const int cr = ur0 + i;
          int sl = 0, ps = 0;
#pragma unroll
          for (int j = 0; j < NJC; ++j) {
            const int a = __shfl_sync(FULL_MASK, cslot[j], cr & 31);
            const int b = __shfl_sync(FULL_MASK, cpos[j], cr & 31);
            if (j == (cr >> 5)) {
              sl = a;
              ps = b;
            }
          }
          const bool valid = i < unr;
          const bool miss = valid && (sl & HS_SLOT_MISS_FLAG) != 0;
          if (i < TILE) {
            tab[i] = miss ? (sl & ~HS_SLOT_MISS_FLAG) : -1;
            mp[i] = miss ? ps : -1;
          }
          usl[m] = (valid && !miss) ? sl : -1;
          hit_rows += __popc(__ballot_sync(FULL_MASK, valid && !miss));
          miss_rows += __popc(__ballot_sync(FULL_MASK, miss));
        }
        __syncwarp();
        if (lane == 0) {
          const int nxt = (u == nunits - 1 && pf_item >= 0) ? (int)(pf_item / NCHK) : -1;
          desc[s] = Desc{DESC_UNIT, r, c, ur0, unr, u == 0 ? 1 : 0, u == nunits - 1 ? 1 : 0, miss_rows, nxt, 0, 0, 0};
          mbar_arrive(&dready[s]);   // the fetcher may read the descriptor and tables now
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&full[s], (uint32_t)(hit_rows * g.row_bytes));
        }
        __syncwarp();
#pragma unroll
        for (int m = 0; m < NJU; ++m) {   // hit rows: one bulk copy each
          const int i = lane + 32 * m;
          int slot = usl[m];
          if (slot < 0) continue;
          if (slot >= g.hot_slots) {   // never expected: keep the copy in bounds
            set_error(p.s.dev_error, HS_DEVERR_METADATA);
            slot = 0;
          }
          bulk_g2s_hint(st_s + (size_t)i * row_stride, hot + (size_t)slot * g.row_bytes, (uint32_t)g.row_bytes,
                        &full[s], stream_policy);
        }
        HS_TRACE_IF(p, 2, 2, lane == 0 && it == 0);
        s = (s + 1 == nstage) ? 0 : s + 1;
        ++it;
        if (u == 0) {   // the next chunk's metadata now, if its request is already published
          const long long nx = (long long)__shfl_sync(FULL_MASK, nxt, 0);
          pf_item = -1;
          pf_warm = false;
          if (nx < total) {
            const int rn = (int)(nx / NCHK);
            unsigned v = 0;
            if (lane == 0) v = ld_acquire(p.s.ready + rn);
            v = __shfl_sync(FULL_MASK, v, 0);
            if (v != 0u) {
              pf.kk = (int)v - 1;
              load_rows(pf, rn, (int)(nx % NCHK));
              pf_item = nx;
            }
          }
        }
        if (pf_item >= 0 && !pf_warm && (u == 1 || u == nunits - 1)) {
          // one unit later (its metadata has landed by now): the next chunk's hit
          // rows start moving into L2, one bulk prefetch per row, so that its bulk
          // copies read L2 and more bytes are in flight than the stages hold
          pf_warm = true;
          const int pr0 = (int)(pf_item % NCHK) * CR;
          const int pnr = max(0, min(CR, pf.kk - pr0));
          const long long rln = (long long)pf.req * g.n_layers + p.layer;
          const unsigned char* hotn =
              reinterpret_cast<const unsigned char*>(p.s.hot) + (size_t)rln * g.hot_slots * g.row_bytes;
#pragma unroll
          for (int j = 0; j < NJC; ++j) {
            const int sl = pf.slot[j];
            if (lane + 32 * j < pnr && !(sl & HS_SLOT_MISS_FLAG) && sl >= 0 && sl < g.hot_slots)
              bulk_prefetch_l2(hotn + (size_t)sl * g.row_bytes, (uint32_t)g.row_bytes);
          }
        }
      }
      cur = (long long)__shfl_sync(FULL_MASK, nxt, 0);
      if (lane == 0 && cur < total) nxt = atomicAdd(&p.s.sync[2], 1u);
      ++n_items;
    }
    // no more work: tell the fetcher and the consumers
    if (!dead && take_stage() && lane == 0) {
      desc[s] = Desc{DESC_STOP, 0, 0, 0, 0, 0, 0, 0, -1, 0, 0, 0};
      mbar_arrive(&dready[s]);
      mbar_arrive(&full[s]);
    }
    __syncwarp();
    HS_TRACE_IF(p, 2, 3, lane == 0);
    if (lane == 0) {
      HS_TRACE_VAL(p, 2, 10, tw_ready);
      HS_TRACE_VAL(p, 2, 11, tw_empty);
      HS_TRACE_VAL(p, 2, 12, (unsigned long long)n_items);
    }
  } else if (warp == PREFETCHER) {
    // =========================== prefetcher warp ===========================
    for (;;) {
      unsigned r = 0;
      if (lane == 0) r = atomicAdd(&p.s.sync[4], 1u);
      r = __shfl_sync(FULL_MASK, r, 0);
      if (r >= (unsigned)p.n_req) break;
      // the resolver's miss list, which it writes before publication; a request
      // published without one (fetch mode 1: RESOLVE pulled its rows) is skipped
      unsigned mc = 0, rd = 0;
      if (lane == 0) {
        const unsigned long long t0 = global_timer_ns();
        unsigned ns = 32;
        for (uint32_t it = 1;; ++it) {
          mc = *reinterpret_cast<volatile const unsigned*>(p.s.miss_cnt + r);
          rd = ld_acquire(p.s.ready + r);
          if (mc != 0u || rd != 0u) break;
          __nanosleep(ns);
          if (ns < 512) ns <<= 1;
          if ((it & 63u) == 0 && global_timer_ns() - t0 > WAIT_LIMIT_NS) break;
        }
        if (mc == 0u && rd != 0u) mc = *reinterpret_cast<volatile const unsigned*>(p.s.miss_cnt + r);
      }
      mc = __shfl_sync(FULL_MASK, mc, 0);
      rd = __shfl_sync(FULL_MASK, rd, 0);
      if ((mc == 0u && rd == 0u) || *abort_flag) break;   // a publication that never came: the loader reports it
      if (mc == 0u) continue;
      const int n = min((int)mc - 1, K);
      const int req = p.req_ids ? p.req_ids[r] : (int)r;
      if (req < 0 || req >= g.max_requests) continue;
      const long long rl = (long long)req * g.n_layers + p.layer;
      const unsigned char* host =
          reinterpret_cast<const unsigned char*>(p.s.host_kv) + (size_t)rl * g.max_context * g.row_bytes;
      const int32_t* mp = p.s.miss_pos + (long long)r * K;
      const int psh = g.page_shift;
      for (int i = lane; i < n; i += 32) {
        const int u = __ldcg(mp + i);   // a missed unit: a position, or a page of 2^psh
        if (u < 0) continue;            // the appended token: its row is not in the host copy yet
        const long long pos0 = (long long)u << psh;
        if (pos0 >= g.max_context) continue;
        const long long nr = min((long long)1 << psh, (long long)g.max_context - pos0);
        bulk_prefetch_l2(host + pos0 * g.row_bytes, (uint32_t)(nr * g.row_bytes));
      }
    }
  } else if (warp == FETCHER) {
    // ============================ fetcher warp ============================
    // Missed rows of each unit, from the mapped host copy straight into their
    // stage rows; the stage's full barrier completes when these copies land.
    unsigned long long n_fetched = 0;
    for (long long it = 0;; ++it) {
      const int s = (int)(it % nstage);
      if (!__all_sync(FULL_MASK, wait_or_abort(&dready[s], (uint32_t)((it / nstage) & 1), abort_flag, p.s.dev_error,
                                               4 * WAIT_LIMIT_NS)))
        break;
      const Desc dsc = desc[s];
      if (dsc.type == DESC_STOP) {
        if (lane == 0) mbar_arrive(&full[s]);
        break;
      }
      const int r = dsc.ri;
      const int req = p.req_ids ? p.req_ids[r] : r;
      const long long rl = (long long)req * g.n_layers + p.layer;
      const unsigned char* host =
          reinterpret_cast<const unsigned char*>(p.s.host_kv) + (size_t)rl * g.max_context * g.row_bytes;
      unsigned char* st_s = stage + (size_t)s * L.stage_bytes;
      const int* mp = mpos + s * TILE_MAX;
      for (int i = 0; i < dsc.nr; ++i) {
        const int ps = mp[i];
        if (ps < 0) continue;
        const unsigned char* src = host + (size_t)ps * g.row_bytes;
        unsigned char* dst = st_s + (size_t)i * row_stride;
        for (int v = lane; v < rvec; v += 32) cp_async_16(dst + v * 16, src + v * 16);
        ++n_fetched;
      }
      cp_async_mbar_arrive(&full[s]);   // balanced: completes when this lane's copies land
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
      if (dsc.nmiss > 0) {
        // once the unit has landed, the fetched rows go on into their hot slots
        // (bulk shared -> global), so later steps hit; the stage is released only
        // after these copies have read it
        if (!__all_sync(FULL_MASK, wait_or_abort(&full[s], (uint32_t)((it / nstage) & 1), abort_flag,
                                                 p.s.dev_error, 4 * WAIT_LIMIT_NS)))
          break;
        const int* tab = slot_tab + s * TILE_MAX;
        unsigned char* hotw = reinterpret_cast<unsigned char*>(p.s.hot) + (size_t)rl * g.hot_slots * g.row_bytes;
        fence_proxy_async_smem();   // cp.async writes -> async-proxy reads
        bool any = false;
        for (int i = lane; i < TILE; i += 32) {
          const int slot = tab[i];
          if (slot >= 0 && slot < g.hot_slots) {
            any = true;
            bulk_s2g(hotw + (size_t)slot * g.row_bytes, st_s + (size_t)i * row_stride, (uint32_t)g.row_bytes);
          }
        }
        if (any) {
          bulk_commit();
          bulk_wait_read_all();
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    cp_async_wait_all();
    bulk_wait_all();   // the hot-slot writes of the fetched rows are complete before the CTA goes on
    if (lane == 0) HS_TRACE_VAL(p, 2, 14, n_fetched);
  } else {
    // ============================ consumer warps ============================
    const int kvh = warp % HKV;
    const int slice = warp / HKV;
    const int gq = lane >> 2, tq = lane & 3;
    const float sl2 = p.scale_log2;
    // Transposed products, so that a unit's 16 rows are the mma's M and the
    // group's query heads its N (8 per n-tile, NT tiles): S^T = K Q^T, then
    // O^T = V^T P^T with P^T moved into the B layout by movmatrix.  With at most
    // 8 heads per kv head that is half the tensor work of heads-as-M.
    constexpr int NT = (G + 7) / 8;
    uint32_t qb[NT][8][2], qn[NT][8][2];   // Q^T as the B operand; qn: the next chunk's, loaded ahead
    int qn_r = -1;
    auto load_q = [&](uint32_t (&qd)[NT][8][2], int r) {
      const uint16_t* qg = p.q + ((long long)r * HQ + kvh * G) * D;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = nt * 8 + gq;   // head (B column) of this lane
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int d0 = ks * 16 + 2 * tq;
          qd[nt][ks][0] = h < G ? *reinterpret_cast<const uint32_t*>(qg + h * D + d0) : 0u;
          qd[nt][ks][1] = h < G ? *reinterpret_cast<const uint32_t*>(qg + h * D + d0 + 8) : 0u;
        }
      }
    };
    float ot[NT][8][4];   // O^T: dims 16m + gq (+8) x heads nt * 8 + 2tq (+1)
    float mh[NT][2], lh[NT][2];   // per head 2tq, 2tq + 1 of each n-tile: running max, partial sum
    int q_r = -1;

    unsigned long long tw_full = 0, t_busy = 0;   // trace builds only
    for (long long it = 0;; ++it) {
      const int s = (int)(it % nstage);
      const unsigned long long t0 = tid == 0 ? global_timer_ns() : 0ull;
      const bool ok = wait_or_abort(&full[s], (uint32_t)((it / nstage) & 1), abort_flag, p.s.dev_error,
                                    4 * WAIT_LIMIT_NS);
      const unsigned long long t1 = tid == 0 ? global_timer_ns() : 0ull;
      const unsigned long long tw = t1 - t0;
      tw_full += tw;
      if (named_sync_or(BAR_VOTE, NCONS * 32, !ok)) break;   // the consumers leave together
      const Desc dsc = desc[s];
      if (tid == 0 && dsc.type == DESC_UNIT) {
        const int k = dsc.nmiss > 0 ? 0 : 2;
        s_wait[k] += tw;
        s_wait[k + 1] += 1;
      }
      if (dsc.type == DESC_STOP) break;
      const int r = dsc.ri;
      if (dsc.first) {
        if (r != q_r) {
          q_r = r;
          if (r == qn_r) {   // loaded during the previous chunk's last unit
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int ks = 0; ks < 8; ++ks) {
                qb[nt][ks][0] = qn[nt][ks][0];
                qb[nt][ks][1] = qn[nt][ks][1];
              }
          } else {
            load_q(qb, r);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int m = 0; m < 8; ++m) ot[nt][m][0] = ot[nt][m][1] = ot[nt][m][2] = ot[nt][m][3] = 0.f;
          mh[nt][0] = mh[nt][1] = -INFINITY;
          lh[nt][0] = lh[nt][1] = 0.f;
        }
      }
      const int nv = max(0, min(ATT_SUBTILE, dsc.nr - slice * ATT_SUBTILE));
      HS_TRACE_IF(p, 2, 4, tid == 0 && it == 0);
      const unsigned char* st_s = stage + (size_t)s * L.stage_bytes;
      if (nv > 0) {
        const int rbase = slice * ATT_SUBTILE;
        // ---- S^T = K Q^T: A = the 16 rows' K (8 k-steps of 16 dims), loaded first ----
        uint32_t fr[8][4];
        {
          const uint32_t rowa =
              smem_addr(st_s + (size_t)(rbase + (lane & 7) + 8 * ((lane >> 3) & 1)) * row_stride);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) ldsm_x4(fr[ks], rowa + (uint32_t)((kvh * D + 16 * ks + 8 * (lane >> 4)) * 2));
        }
        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float sx[4] = {0.f, 0.f, 0.f, 0.f};   // two accumulation chains
          sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
          for (int ks = 0; ks < 8; ks += 2) {
            mma_bf16(sc[nt], fr[ks], qb[nt][ks][0], qb[nt][ks][1]);
            mma_bf16(sx, fr[ks + 1], qb[nt][ks + 1][0], qb[nt][ks + 1][1]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[nt][e] += sx[e];
        }
        // ---- online softmax per head (a column: rows gq, gq + 8 of the 8 lanes with this tq);
        // rows >= nv are masked out ----
        const bool ok0 = gq < nv, ok1 = gq + 8 < nv;
        uint32_t pt[NT][2];   // P^T as the B operand (rows 0-7 | 8-15 x head gq)
        bool rescale = false;
        float al[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float mx[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            sc[nt][e] = ok0 ? sc[nt][e] * sl2 : -INFINITY;
            sc[nt][2 + e] = ok1 ? sc[nt][2 + e] * sl2 : -INFINITY;
            mx[e] = fmaxf(sc[nt][e], sc[nt][2 + e]);
            mx[e] = fmaxf(mx[e], __shfl_xor_sync(FULL_MASK, mx[e], 4));
            mx[e] = fmaxf(mx[e], __shfl_xor_sync(FULL_MASK, mx[e], 8));
            mx[e] = fmaxf(mx[e], __shfl_xor_sync(FULL_MASK, mx[e], 16));
            // padded heads (>= G) see all-zero scores, never -inf: every m stays finite
            const float mn = fmaxf(mh[nt][e], mx[e]);
            al[nt][e] = exp2f(mh[nt][e] - mn);   // -inf - x -> 0
            mh[nt][e] = mn;
            rescale |= al[nt][e] != 1.f;
          }
          const float p0 = exp2f(sc[nt][0] - mh[nt][0]), p1 = exp2f(sc[nt][1] - mh[nt][1]);
          const float p2 = exp2f(sc[nt][2] - mh[nt][0]), p3 = exp2f(sc[nt][3] - mh[nt][1]);
          lh[nt][0] = lh[nt][0] * al[nt][0] + (p0 + p2);
          lh[nt][1] = lh[nt][1] * al[nt][1] + (p1 + p3);
          pt[nt][0] = movmatrix_trans(pack_bf16(p0, p1));   // rows 0-7
          pt[nt][1] = movmatrix_trans(pack_bf16(p2, p3));   // rows 8-15
        }
        if (__any_sync(FULL_MASK, rescale)) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              ot[nt][m][0] *= al[nt][0];
              ot[nt][m][1] *= al[nt][1];
              ot[nt][m][2] *= al[nt][0];
              ot[nt][m][3] *= al[nt][1];
            }
        }
        // ---- O^T += V^T P^T: A = V^T of 16 dims x the 16 rows (ldmatrix .trans), loaded first ----
        {
          const uint32_t rowv =
              smem_addr(st_s + (size_t)(rbase + (lane & 7) + 8 * (lane >> 4)) * row_stride);
#pragma unroll
          for (int m = 0; m < 8; ++m)
            ldsm_x4_t(fr[m], rowv + (uint32_t)((g.v_off + kvh * D + 16 * m + 8 * ((lane >> 3) & 1)) * 2));
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int m = 0; m < 8; ++m) mma_bf16(ot[nt][m], fr[m], pt[nt][0], pt[nt][1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      t_busy += HS_TNOW() - t1;
      if (NT == 1 && dsc.last && dsc.nxt >= 0 && dsc.nxt != r && dsc.nxt != qn_r) {   // the next chunk's query, ahead
        load_q(qn, dsc.nxt);
        qn_r = dsc.nxt;
      }
      if (dsc.last) {   // the chunk's partial (m, l, o) for this slice
        const int part = dsc.c * NSLICE + slice;
        float* po = p.s.part_o + ((long long)r * NPARTS + part) * HQ * D;
        float* pml = p.s.part_ml + ((long long)r * NPARTS + part) * HQ * 2;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float l = lh[nt][e];   // the sum over all 16 rows: this lane holds rows gq, gq + 8
            l += __shfl_xor_sync(FULL_MASK, l, 4);
            l += __shfl_xor_sync(FULL_MASK, l, 8);
            l += __shfl_xor_sync(FULL_MASK, l, 16);
            const int hl = nt * 8 + 2 * tq + e;   // head within the group
            if (hl < G) {
              float* ph = po + (long long)(kvh * G + hl) * D;
#pragma unroll
              for (int m = 0; m < 8; ++m) {
                ph[16 * m + gq] = ot[nt][m][e];
                ph[16 * m + gq + 8] = ot[nt][m][2 + e];
              }
              if (gq == 0) *reinterpret_cast<float2*>(pml + (kvh * G + hl) * 2) = make_float2(mh[nt][e], l);
            }
          }
        // every consumer warp has written its part of the chunk: count it done
        named_sync(BAR_CHUNK, NCONS * 32);
        if (tid == 0) {
          __threadfence();
          red_release_add(p.s.att_done + r, 1u);
        }
      }
    }
    HS_TRACE_IF(p, 2, 5, tid == 0);
    if (tid == 0) {
      HS_TRACE_VAL(p, 2, 13, tw_full);
      HS_TRACE_VAL(p, 2, 15, s_wait[0]);
      HS_TRACE_VAL(p, 2, 16, s_wait[1]);
      HS_TRACE_VAL(p, 2, 17, t_busy);
    }
  }

  __syncthreads();
  const bool aborted = *abort_flag != 0;
  if (aborted) {
    // drain copies that may still be in flight (bounded) before the buffers go away
    if (tid == 0) {
      for (int s2 = 0; s2 < nstage; ++s2) {
        (void)mbar_wait_bounded(&full[s2], 0);
        (void)mbar_wait_bounded(&full[s2], 1);
      }
    }
    __syncthreads();
  }

  // ---- merge: (request, group of MERGE_HEADS heads) items in request order,
  // each once every chunk of its request is written; the stage memory is free now
  __shared__ int s_item, s_ok;
  constexpr int HPM = HQ < MERGE_HEADS ? HQ : MERGE_HEADS;
  constexpr int NHG = HQ / HPM;
  float* wsm = reinterpret_cast<float*>(stage);   // [parts][HPM] merge weights
  float* Ms = wsm + (size_t)NPARTS * HPM;          // [HPM]
  float* Ls = Ms + HPM;                            // [HPM]
  while (!aborted) {
    if (tid == 0) s_item = (int)atomicAdd(&p.s.sync[5], 1u);
    __syncthreads();
    const int item = s_item;
    if (item >= p.n_req * NHG) break;
    const int r = item / NHG, h0 = (item % NHG) * HPM;
    if (tid == 0) {
      // a chunk of this request may sit behind a chunk whose own request was
      // never published (its loader gives up after WAIT_LIMIT_NS and goes on), so
      // this wait outlasts that one
      s_ok = wait_counter(p.s.att_done + r, (unsigned)NCHK, 4 * WAIT_LIMIT_NS) ? 1 : 0;
      if (!s_ok) set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
    }
    __syncthreads();
    const int rdy = (int)__ldcg(p.s.ready + r);
    const int kk = max(0, rdy - 1);
    const int nparts = ((kk + CR - 1) / CR) * NSLICE;
    uint16_t* outp = p.out + ((long long)r * HQ + h0) * D;
    if (!s_ok || nparts == 0) {   // nothing selected (or never published): the output is defined as 0
      for (int e = tid; e < HPM * D; e += THREADS) outp[e] = 0;
      __syncthreads();
      continue;
    }
    const float* pml = p.s.part_ml + (long long)r * NPARTS * HQ * 2;
    const float* po = p.s.part_o + (long long)r * NPARTS * HQ * D;
    // per head (one warp each): M = max_q m_q, w_q = 2^(m_q - M), L = sum_q w_q l_q
    if (warp < HPM) {
      const int h = h0 + warp;
      float mx = -INFINITY;
      for (int q = lane; q < nparts; q += 32) mx = fmaxf(mx, __ldcg(pml + ((long long)q * HQ + h) * 2));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, o));
      float l = 0.f;
      for (int q = lane; q < nparts; q += 32) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(pml) + (long long)q * HQ + h);
        const float w = exp2f(ml.x - mx);
        wsm[q * HPM + warp] = w;
        l = fmaf(ml.y, w, l);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(FULL_MASK, l, o);
      if (lane == 0) {
        Ms[warp] = mx;
        Ls[warp] = l;
      }
    }
    __syncthreads();
    // out = (sum_q w_q o_q) / L, parts in order, one float4 of a head's dims per thread
    if (tid < HPM * (D / 4)) {
      const int hh = tid / (D / 4), d4 = tid % (D / 4);
      const float4* col = reinterpret_cast<const float4*>(po + (long long)(h0 + hh) * D) + d4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      constexpr int UQ = 8;   // parts in flight per thread
      for (int q = 0; q < nparts; q += UQ) {
        float4 v[UQ];
#pragma unroll
        for (int u = 0; u < UQ; ++u)
          v[u] = q + u < nparts ? __ldcg(col + (long long)(q + u) * HQ * D / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < UQ; ++u)
          if (q + u < nparts) {
            const float w = wsm[(q + u) * HPM + hh];
            acc.x = fmaf(w, v[u].x, acc.x);
            acc.y = fmaf(w, v[u].y, acc.y);
            acc.z = fmaf(w, v[u].z, acc.z);
            acc.w = fmaf(w, v[u].w, acc.w);
          }
      }
      const float inv = 1.f / Ls[hh];
      uint2 packed;
      packed.x = pack_bf16(acc.x * inv, acc.y * inv);
      packed.y = pack_bf16(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(outp + (long long)hh * D + 4 * d4) = packed;
    }
    __syncthreads();   // wsm, Ms, Ls and s_item are reused
  }

  // the last CTA to leave resets the call's queues, counters and flags (every
  // CTA has taken its last item and merged its last request by then)
  __shared__ int s_last;
  if (tid == 0) {
    if (s_wait[1]) {
      red_add_u64(&p.s.glob[4], s_wait[0]);
      red_add_u64(&p.s.glob[5], s_wait[1]);
    }
    if (s_wait[3]) {
      red_add_u64(&p.s.glob[6], s_wait[2]);
      red_add_u64(&p.s.glob[7], s_wait[3]);
    }
    if ((int)blockIdx.x < p.att_grid) {
      p.s.att_cta[2 * blockIdx.x] = s_wait[4];
      p.s.att_cta[2 * blockIdx.x + 1] = global_timer_ns();
    }
    const unsigned prev = atom_acq_rel_add(&p.s.sync[3], 1u);
    s_last = prev + 1 == gridDim.x;
  }
  __syncthreads();
  if (s_last) {
    for (int r = tid; r < p.n_req; r += THREADS) {
      p.s.ready[r] = 0;
      p.s.miss_cnt[r] = 0;
      p.s.att_done[r] = 0;
    }
    if (tid == 0) {
      p.s.sync[2] = 0;
      p.s.sync[3] = 0;
      p.s.sync[4] = 0;
      p.s.sync[5] = 0;
    }
  }
  HS_TRACE(p, 2, 6);
  // complete only after the select kernel has: the next launch on the stream
  // then sees both kernels finished
  griddep_wait();
}

// Combines the partials of each (request, head) in part order: grid (heads /
// heads-per-CTA, requests), DV / 4 threads per head, one float4 of the head's
// output dims per thread.  out = sum_q 2^(m_q - M) o_q / sum_q 2^(m_q - M) l_q.
// Part counts are per group of GH heads (GQA: one group; latent rows: 16 heads).
constexpr int MERGE_MAX_PARTS = 1024;

template <int HQ, int DV, int GH>
__global__ void __launch_bounds__(128) attn_merge_kernel(DecodeParams p) {
  constexpr int TPH = DV / 4;                                        // threads per head
  constexpr int HPC = (128 / TPH) < HQ ? (128 / TPH) : HQ;           // heads per CTA
  __shared__ float2 mls[MERGE_MAX_PARTS / 8][HPC];   // (m, l) of a batch of parts
  __shared__ float wsm[MERGE_MAX_PARTS][HPC];
  __shared__ float Ms[HPC], Ls[HPC];
  const int tid = threadIdx.x;
  const int ri = blockIdx.y;
  const int h0 = blockIdx.x * HPC;
  griddep_wait();   // the attention kernel's partials
  griddep_launch_dependents();
  const int nparts = p.s.att_nparts[(long long)ri * (HQ / GH) + h0 / GH];
  if (!p.g.shared_kv && blockIdx.x == 0 && tid == 0) {   // this call is done with the request
    p.s.ready[ri] = 0;
    p.s.miss_cnt[ri] = 0;
  }
  if (nparts <= 0) {   // nothing selected: the output is defined as 0
    if (!p.g.shared_kv)
      for (int e = tid; e < HPC * DV; e += blockDim.x) p.out[((long long)ri * HQ + h0) * DV + e] = 0;
    return;
  }
  if (nparts > MERGE_MAX_PARTS) {   // not reachable with the shapes hs_create accepts
    if (tid == 0) set_error(p.s.dev_error, HS_DEVERR_METADATA);
    return;
  }
  const float* pml = p.s.part_ml + (long long)ri * p.att_parts * HQ * 2;
  const float* po = p.s.part_o + (long long)ri * p.att_parts * HQ * DV;
  // weights: M = max_q m_q, w_q = 2^(m_q - M), L = sum_q w_q l_q (one thread per head, parts in order)
  if (tid < HPC) {
    Ms[tid] = -INFINITY;
    Ls[tid] = 0.f;
  }
  for (int q0 = 0; q0 < nparts; q0 += MERGE_MAX_PARTS / 8) {
    const int nq = min(MERGE_MAX_PARTS / 8, nparts - q0);
    __syncthreads();
    for (int e = tid; e < nq * HPC; e += blockDim.x)
      mls[e / HPC][e % HPC] =
          __ldcg(reinterpret_cast<const float2*>(pml) + (long long)(q0 + e / HPC) * HQ + h0 + e % HPC);
    __syncthreads();
    if (tid < HPC)
      for (int q = 0; q < nq; ++q) Ms[tid] = fmaxf(Ms[tid], mls[q][tid].x);
  }
  __syncthreads();
  for (int q0 = 0; q0 < nparts; q0 += MERGE_MAX_PARTS / 8) {
    const int nq = min(MERGE_MAX_PARTS / 8, nparts - q0);
    for (int e = tid; e < nq * HPC; e += blockDim.x)
      mls[e / HPC][e % HPC] =
          __ldcg(reinterpret_cast<const float2*>(pml) + (long long)(q0 + e / HPC) * HQ + h0 + e % HPC);
    __syncthreads();
    if (tid < HPC)
      for (int q = 0; q < nq; ++q) {
        const float w = exp2f(mls[q][tid].x - Ms[tid]);
        wsm[q0 + q][tid] = w;
        Ls[tid] = fmaf(mls[q][tid].y, w, Ls[tid]);
      }
    __syncthreads();
  }
  const int hh = tid / TPH;   // head within this CTA
  if (hh >= HPC) return;
  const int d4 = tid % TPH;   // float4 of the head's output dims
  const float inv = 1.f / Ls[hh];
  const float4* col = reinterpret_cast<const float4*>(po + (long long)(h0 + hh) * DV) + d4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int UQ = 8;   // parts in flight per thread
  for (int q = 0; q < nparts; q += UQ) {
    float4 v[UQ];
#pragma unroll
    for (int u = 0; u < UQ; ++u)
      v[u] = q + u < nparts ? __ldcg(col + (long long)(q + u) * HQ * DV / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < UQ; ++u)
      if (q + u < nparts) {
        const float w = wsm[q + u][hh] * inv;
        acc.x = fmaf(v[u].x, w, acc.x);
        acc.y = fmaf(v[u].y, w, acc.y);
        acc.z = fmaf(v[u].z, w, acc.z);
        acc.w = fmaf(v[u].w, w, acc.w);
      }
  }
  uint2 pk;
  pk.x = pack_bf16(acc.x, acc.y);
  pk.y = pack_bf16(acc.z, acc.w);
  *reinterpret_cast<uint2*>(p.out + ((long long)ri * HQ + h0 + hh) * DV + 4 * d4) = pk;
}

template <int HQ, int DV, int GH>
static cudaError_t run_merge(const DecodeParams* p, cudaStream_t st) {
  constexpr int TPH = DV / 4;
  constexpr int HPC = (128 / TPH) < HQ ? (128 / TPH) : HQ;
  if (p == nullptr) return allow_smem(attn_merge_kernel<HQ, DV, GH>, 0);
  return launch_pdl(attn_merge_kernel<HQ, DV, GH>, dim3(HQ / HPC, p->n_req), dim3(HPC * TPH), 0, st, *p);
}

// p == nullptr: set-up only
static cudaError_t dispatch_merge(const Geometry& g, const DecodeParams* p, cudaStream_t st) {
  if (g.shared_kv) {   // part counts per item head group: 16 heads at h_q = 16, else 32
    switch (g.h_q) {
      case 16: return run_merge<16, 512, 16>(p, st);
      case 32: return run_merge<32, 512, 32>(p, st);
      case 64: return run_merge<64, 512, 32>(p, st);
      case 128: return run_merge<128, 512, 32>(p, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (g.h_q) {
    case 1: return run_merge<1, 128, 1>(p, st);
    case 2: return run_merge<2, 128, 2>(p, st);
    case 4: return run_merge<4, 128, 4>(p, st);
    case 8: return run_merge<8, 128, 8>(p, st);
    case 16: return run_merge<16, 128, 16>(p, st);
    case 32: return run_merge<32, 128, 32>(p, st);
    case 64: return run_merge<64, 128, 64>(p, st);
    case 128: return run_merge<128, 128, 128>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_merge(const DecodeParams& p, cudaStream_t st) { return dispatch_merge(p.g, &p, st); }

template <int G, int HKV>
static cudaError_t run_gqa(const DecodeParams* p, size_t smem, cudaStream_t st) {
  auto kern = attn_gqa_kernel<G, HKV>;
  if (p == nullptr)   // prepare: allow the shared memory this shape needs
    return allow_smem(kern, smem);
  const int ns = attention_stages(p->g, 227 * 1024);
  return launch_pdl(kern, dim3(p->att_grid), dim3(THREADS), smem, st, *p, ns);   // merges its own partials
}

template <int HKV>
static cudaError_t dispatch_g(const Geometry& g, const DecodeParams* p, size_t smem, cudaStream_t st) {
  switch (g.h_q / HKV) {
    case 1: return run_gqa<1, HKV>(p, smem, st);
    case 2: return run_gqa<2, HKV>(p, smem, st);
    case 4: return run_gqa<4, HKV>(p, smem, st);
    case 8: return run_gqa<8, HKV>(p, smem, st);
    case 16: return run_gqa<16, HKV>(p, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

static cudaError_t dispatch(const Geometry& g, const DecodeParams* p, size_t smem, cudaStream_t st) {
  switch (g.h_kv) {
    case 1: return dispatch_g<1>(g, p, smem, st);
    case 2: return dispatch_g<2>(g, p, smem, st);
    case 4: return dispatch_g<4>(g, p, smem, st);
    case 8: return dispatch_g<8>(g, p, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t prepare_attention(const Geometry& g, size_t smem) {
  const cudaError_t e = g.shared_kv ? dispatch_mla(g, nullptr, smem, 0) : dispatch(g, nullptr, smem, 0);
  return e != cudaSuccess ? e : dispatch_merge(g, nullptr, 0);
}

cudaError_t launch_attention(const DecodeParams& p, size_t smem, cudaStream_t st) {
  return p.g.shared_kv ? dispatch_mla(p.g, &p, smem, st) : dispatch(p.g, &p, smem, st);
}

}  // namespace hs
