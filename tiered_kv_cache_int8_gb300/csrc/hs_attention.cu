// Sparse attention over the selected rows (GQA, head dim 128): a persistent,
// warp-specialised flash-decode kernel whose per-request partial results are
// merged in a fixed order by the last CTA that touched the request.
//
// Method: "Heterogeneous LLM Serving with General-Purpose Processing-Near-Memory
// for Retrieval-Based Sparse Attention" (vsvnakers.github.io), "核心公式与算法",
// formula 2: softmax(Q K^T / sqrt(d_k), masked to the retrieved entries) V —
// read as a softmax over the selected positions only.  "KV卸载上主机:
// HiSparse、PDD与DDR4回收", "论文1：HiSparse": the attention math is unchanged
// by the cache, so the result must not depend on where the rows sit.
//
// Design (sm_103a).  The kernel is HBM-bound (each K/V byte is used by the
// h_q / h_kv query heads of its group only), so the goal is to keep enough
// bytes in flight on every SM with as few instructions per byte as possible:
//  * Persistent grid, one CTA per SM.  The selected rows of all requests are
//    flattened into units of TILE rows (16 rows per warp slice); CTA c takes
//    units [c*U/G, (c+1)*U/G).  The split depends only on the k_eff of each
//    request and on the grid size, never on B or on slot placement.
//  * Warp specialisation: warp 8 is the producer.  For each unit it copies every
//    selected row (all kv heads: one contiguous hot slot) HBM -> shared memory
//    with one 1-D bulk async copy (cp.async.bulk, mbarrier completion) into a
//    row-padded layout (16 extra bytes per row put the 8 rows of an ldmatrix
//    phase in 8 different bank groups); up to 4 stages with full/empty mbarriers.
//  * Warps 0-7 consume: warp w serves kv head w % h_kv and row slice w / h_kv.
//    S = Q K^T and O += P V run on mma.sync m16n8k16 (bf16 in, fp32 accumulate)
//    with the group's query heads as the 16 M rows (zero-padded).  The tensor
//    cores are used to cut the instruction count per byte, not for throughput;
//    K and V fragments come straight from shared memory with ldmatrix (.trans
//    for V).  Online softmax in fp32 (exp2, scale * log2(e) applied to the fp32
//    scores); P enters the second product as bf16.
//  * Every (CTA, request, slice) writes a partial (m, l, o) to scratch; the last
//    CTA to finish a request (arrival counter) merges its partials in CTA order
//    and writes bf16.  Rows are visited in ascending selection order and the
//    merge order is fixed, so the output is bit-identical for any B.
#include <cuda_bf16.h>

#include "hs_internal.cuh"

namespace hs {

namespace {

constexpr int D = 128;
constexpr int NCONS = 8;                   // consumer warps
constexpr int NLOAD = 2;                   // loader warps (host fetch of missed rows)
constexpr int PRODUCER = NCONS;            // warp index of the producer
constexpr int THREADS = (NCONS + 1 + NLOAD) * 32;
constexpr int MAX_STAGES = 4;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct AttLayout {
  size_t bar, mlist, prefix, stage, stage_bytes, total;
};

// Shared memory: barriers and flags | unit prefix of every request | stages.
__host__ __device__ inline AttLayout att_layout(const Geometry& g, int nstage) {
  AttLayout L;
  const int nslice = NCONS / g.h_kv;
  const int tile = ATT_SUBTILE * nslice;
  size_t off = 0;
  L.bar = off;
  off += 256;   // full[4], empty[4], abort flag, loaded-unit count, miss-list count
  L.mlist = off;
  off += align_up((size_t)tile * 4, 128);   // the loader's miss list of one unit
  L.prefix = off;
  off += align_up((size_t)(g.max_requests + 1) * 4, 128);
  L.stage = off;
  L.stage_bytes = align_up((size_t)tile * (g.row_bytes + ATT_ROW_PAD), 128);
  off += (size_t)nstage * L.stage_bytes;
  L.total = off;
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

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bounded wait that also gives up once another warp has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
        *abort_flag = 1;
        set_error(err, HS_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void st_release(volatile int* p, int v) {
  asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(smem_addr((const void*)p)), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire(volatile int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_addr((const void*)p)) : "memory");
  return v;
}

// Barrier 1 over the loader warps, returning the OR of `pred` over them.
__device__ __forceinline__ bool loader_bar_or(bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((int)pred), "n"(NLOAD * 32)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// CTA owning flattened unit u when U units are split over G CTAs as [c*U/G, (c+1)*U/G).
__device__ __forceinline__ int owner_of(long long u, long long U, int G) {
  return (int)(((u + 1) * G + U - 1) / U) - 1;
}

}  // namespace

int attention_parts(const Geometry& g) {
  const int nslice = NCONS / g.h_kv;
  const int tile = ATT_SUBTILE * nslice;
  const int units = (g.top_k + tile - 1) / tile;
  return (units + 1) * nslice;
}

static int attention_stages(const Geometry& g, size_t limit) {
  for (int ns = MAX_STAGES; ns >= 2; --ns)
    if (att_layout(g, ns).total <= limit) return ns;
  return 2;
}

size_t attention_smem_bytes(const Geometry& g) { return att_layout(g, attention_stages(g, 227 * 1024)).total; }

template <int G, int HKV>
__global__ void __launch_bounds__(THREADS, 1) attn_gqa_kernel(DecodeParams p, int nstage) {
  constexpr int NSLICE = NCONS / HKV;
  constexpr int TILE = ATT_SUBTILE * NSLICE;
  constexpr int HQ = HKV * G;
  const Geometry& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = g.top_k;
  const int c = blockIdx.x;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  const AttLayout L = att_layout(g, nstage);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + L.bar);
  uint64_t* empty = full + MAX_STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + L.bar + 128);
  volatile int* loaded = reinterpret_cast<volatile int*>(smem_raw + L.bar + 132);   // units fetched
  volatile int* mcount = reinterpret_cast<volatile int*>(smem_raw + L.bar + 136);   // [2], per unit parity
  int* mlist = reinterpret_cast<int*>(smem_raw + L.mlist);
  int* prefix = reinterpret_cast<int*>(smem_raw + L.prefix);   // prefix[i] = first unit of request i
  unsigned char* stage = smem_raw + L.stage;
  const int row_stride = g.row_bytes + ATT_ROW_PAD;
  __shared__ int scan_tmp[THREADS / 32 + 1];
  __shared__ int s_last[2];

  // ---- flattened work list: units of every request (k_eff / TILE, rounded up) ----
  int carry = 0;
  for (int base = 0; base < p.n_req; base += THREADS) {
    const int i = base + tid;
    int units = 0;
    if (i < p.n_req) {
      const int req = p.req_ids ? p.req_ids[i] : i;
      int kk = 0;
      if (req >= 0 && req < g.max_requests) kk = min(K, p.s.length[(long long)req * g.n_layers + p.layer]);
      units = (kk + TILE - 1) / TILE;
      if (kk == 0 && i % (int)gridDim.x == c) {   // nothing selected: the output is defined as 0
        uint16_t* out = p.out + (long long)i * HQ * D;
        for (int e = 0; e < HQ * D; ++e) out[e] = 0;
        if (req >= 0 && req < g.max_requests) set_error(p.s.dev_error, HS_DEVERR_EMPTY);
      }
    }
    int tot;
    const int ex = block_exclusive_scan<THREADS>(units, scan_tmp, &tot);
    if (i < p.n_req) prefix[i] = carry + ex;
    carry += tot;
  }
  if (tid == 0) {
    prefix[p.n_req] = carry;
    for (int s = 0; s < nstage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCONS);
    }
    *abort_flag = 0;
    *loaded = 0;
    mcount[0] = 0;
    mcount[1] = 0;
    fence_mbar_init();
  }
  // Zero the stages once: rows past the end of a request are never copied, and
  // their (masked, weight-0) values must be finite.
  for (size_t e = (size_t)tid * 16; e < (size_t)nstage * L.stage_bytes; e += (size_t)THREADS * 16)
    *reinterpret_cast<int4*>(stage + e) = make_int4(0, 0, 0, 0);
  __syncthreads();
  const long long U = carry;
  // Only the first min(grid, U) CTAs take part, so every taking part owns at
  // least one unit (the arrival counts below rely on that).
  const int Gc = (int)min((long long)gridDim.x, U);
  if (c >= Gc) return;
  const long long u0 = (long long)c * U / Gc, u1 = (long long)(c + 1) * U / Gc;

  // first request with units at or after u0: the last i with prefix[i] <= u0 < prefix[i+1]
  int ri = 0;
  {
    int lo = 0, hi = p.n_req - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= u0) lo = mid;
      else hi = mid - 1;
    }
    ri = lo;
    while (prefix[ri + 1] <= u0) ++ri;
  }

  if (warp == PRODUCER) {
    // ============================ producer warp ============================
    int r = ri;
    int s = 0;
    long long it = 0;
    for (long long u = u0; u < u1; ++u, ++it) {
      while (prefix[r + 1] <= u) ++r;
      const int req = p.req_ids ? p.req_ids[r] : r;
      const long long rl = (long long)req * g.n_layers + p.layer;
      const int kk = min(K, p.s.length[rl]);
      const int row0 = (int)(u - prefix[r]) * TILE;
      const int nr = min(TILE, kk - row0);
      if (it >= nstage) {
        if (!wait_or_abort(&empty[s], (uint32_t)(((it / nstage) + 1) & 1), abort_flag, p.s.dev_error)) break;
      }
      const int32_t* sos = p.s.slot_of_sel + (long long)r * K + row0;
      int slots[TILE / 32 > 0 ? TILE / 32 : 1];
      bool miss = false;
#pragma unroll
      for (int j = 0; j < (TILE + 31) / 32; ++j) {
        const int i = lane + 32 * j;
        slots[j] = i < nr ? sos[i] : 0;
        miss |= (slots[j] & HS_SLOT_MISS_FLAG) != 0;
      }
      if (__any_sync(FULL_MASK, miss)) {
        // the loader warps copy this unit's missed rows into their slots first
        const unsigned long long t_start = global_timer_ns();
        bool ok = true;
        for (uint32_t spin = 0; ld_acquire(loaded) < it + 1; ++spin) {
          if ((spin & 255u) == 0 && (*abort_flag || global_timer_ns() - t_start > WAIT_LIMIT_NS)) {
            if (!*abort_flag && lane == 0) set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
        }
        if (!__all_sync(FULL_MASK, ok)) break;
        fence_proxy_async_global();
      }
      if (lane == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&full[s], (uint32_t)(nr * g.row_bytes));
      }
      __syncwarp();
      const unsigned char* hot =
          reinterpret_cast<const unsigned char*>(p.s.hot) + (size_t)rl * g.hot_slots * g.row_bytes;
#pragma unroll
      for (int j = 0; j < (TILE + 31) / 32; ++j) {
        const int i = lane + 32 * j;
        if (i < nr) {
          int slot = slots[j] & ~HS_SLOT_MISS_FLAG;
          if (slot < 0 || slot >= g.hot_slots) {   // never expected: keep the copy in bounds
            set_error(p.s.dev_error, HS_DEVERR_METADATA);
            slot = 0;
          }
          bulk_g2s(stage + (size_t)s * L.stage_bytes + (size_t)i * row_stride, hot + (size_t)slot * g.row_bytes,
                   (uint32_t)g.row_bytes, &full[s]);
        }
      }
      s = (s + 1 == nstage) ? 0 : s + 1;
    }
  } else if (warp > PRODUCER) {
    // ===================== loader warps: host fetch of missed rows =====================
    // For each unit in order: list the rows RESOLVE flagged as misses, copy them
    // from the mapped pinned host copy into their hot slots (16-byte loads, 8 in
    // flight per thread), make the writes visible to the bulk-copy proxy, then
    // publish the unit count the producer waits on.
    const int lt = (warp - PRODUCER - 1) * 32 + lane;
    constexpr int NLT = NLOAD * 32;
    const int rvec = g.row_bytes / 16;
    int r = ri;
    long long it = 0;
    for (long long u = u0; u < u1; ++u, ++it) {
      while (prefix[r + 1] <= u) ++r;
      const int req = p.req_ids ? p.req_ids[r] : r;
      const long long rl = (long long)req * g.n_layers + p.layer;
      const int kk = min(K, p.s.length[rl]);
      const int row0 = (int)(u - prefix[r]) * TILE;
      const int nr = min(TILE, kk - row0);
      const int32_t* sos = p.s.slot_of_sel + (long long)r * K + row0;
      const int32_t* selp = p.s.sel + (long long)r * K + row0;
      volatile int* cnt = mcount + (it & 1);
      for (int i = lt; i < nr; i += NLT)
        if (sos[i] & HS_SLOT_MISS_FLAG) mlist[atomicAdd((int*)cnt, 1)] = i;
      asm volatile("bar.sync 1, %0;" ::"n"(NLT) : "memory");
      const int nm = *cnt;
      // the other counter was last read before the barrier above and is next
      // written after the barrier below
      if (lt == 0) mcount[(it + 1) & 1] = 0;
      if (nm > 0) {
        const unsigned char* src = reinterpret_cast<const unsigned char*>(p.s.host_kv) +
                                   (size_t)rl * g.max_context * g.row_bytes;
        unsigned char* dst = reinterpret_cast<unsigned char*>(p.s.hot) + (size_t)rl * g.hot_slots * g.row_bytes;
        const int total = nm * rvec;
        constexpr int U = 8;
        for (int e0 = lt; e0 < total; e0 += U * NLT) {
          int4 v[U];
#pragma unroll
          for (int q = 0; q < U; ++q) {
            const int e = e0 + q * NLT;
            if (e < total) {
              const int row = mlist[e / rvec];
              v[q] = ld_nc_v4(src + (size_t)selp[row] * g.row_bytes + (e % rvec) * 16);
            }
          }
#pragma unroll
          for (int q = 0; q < U; ++q) {
            const int e = e0 + q * NLT;
            if (e < total) {
              const int row = mlist[e / rvec];
              const int slot = sos[row] & ~HS_SLOT_MISS_FLAG;
              if (slot >= 0 && slot < g.hot_slots)
                *reinterpret_cast<int4*>(dst + (size_t)slot * g.row_bytes + (e % rvec) * 16) = v[q];
            }
          }
        }
        fence_proxy_async_global();
      }
      // every loader thread's copies of this unit are done: publish (and agree on abort)
      const bool stop = loader_bar_or(*abort_flag != 0);
      if (lt == 0) st_release(loaded, (int)(it + 1));
      if (stop) break;
    }
  } else {
    // ============================ consumer warps ============================
    const int kvh = warp % HKV;
    const int slice = warp / HKV;
    const int gq = lane >> 2, tq = lane & 3;
    const float sl2 = p.scale_log2;
    uint32_t qa[8][4];
    float o[16][4];
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;   // heads gq and gq + 8
    int r = -1;
    int s = 0;

    auto flush = [&](int req_i) {   // partial (m, l, o) of this (CTA, request, slice)
      float ll = l_lo + __shfl_xor_sync(FULL_MASK, l_lo, 1);
      ll += __shfl_xor_sync(FULL_MASK, ll, 2);
      float lh = l_hi + __shfl_xor_sync(FULL_MASK, l_hi, 1);
      lh += __shfl_xor_sync(FULL_MASK, lh, 2);
      const int c_first = owner_of(prefix[req_i], U, Gc);
      const int part = (c - c_first) * NSLICE + slice;
      float* po = p.s.part_o + ((long long)req_i * p.att_parts + part) * HQ * D;
      float* pml = p.s.part_ml + ((long long)req_i * p.att_parts + part) * HQ * 2;
      const int h_lo = kvh * G + gq, h_hi = kvh * G + gq + 8;
      if (gq < G) {
#pragma unroll
        for (int t = 0; t < 16; ++t)
          *reinterpret_cast<float2*>(po + (long long)h_lo * D + 8 * t + 2 * tq) = make_float2(o[t][0], o[t][1]);
        if (tq == 0) {
          pml[h_lo * 2 + 0] = m_lo;
          pml[h_lo * 2 + 1] = ll;
        }
      }
      if (gq + 8 < G) {
#pragma unroll
        for (int t = 0; t < 16; ++t)
          *reinterpret_cast<float2*>(po + (long long)h_hi * D + 8 * t + 2 * tq) = make_float2(o[t][2], o[t][3]);
        if (tq == 0) {
          pml[h_hi * 2 + 0] = m_hi;
          pml[h_hi * 2 + 1] = lh;
        }
      }
    };

    long long it = 0;
    for (long long u = u0; u < u1; ++u, ++it) {
      int rn = r < 0 ? ri : r;
      while (prefix[rn + 1] <= u) ++rn;
      if (rn != r) {
        if (r >= 0) flush(r);
        r = rn;
        // the group's query heads as the mma A operand (rows >= G are zero)
        const uint16_t* qg = p.q + ((long long)r * HQ + kvh * G) * D;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int d0 = ks * 16 + 2 * tq;
          qa[ks][0] = gq < G ? *reinterpret_cast<const uint32_t*>(qg + gq * D + d0) : 0u;
          qa[ks][1] = gq + 8 < G ? *reinterpret_cast<const uint32_t*>(qg + (gq + 8) * D + d0) : 0u;
          qa[ks][2] = gq < G ? *reinterpret_cast<const uint32_t*>(qg + gq * D + d0 + 8) : 0u;
          qa[ks][3] = gq + 8 < G ? *reinterpret_cast<const uint32_t*>(qg + (gq + 8) * D + d0 + 8) : 0u;
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
        m_lo = m_hi = -INFINITY;
        l_lo = l_hi = 0.f;
      }
      const int req = p.req_ids ? p.req_ids[r] : r;
      const int kk = min(K, p.s.length[(long long)req * g.n_layers + p.layer]);
      const int row0 = (int)(u - prefix[r]) * TILE;
      const int nv = max(0, min(ATT_SUBTILE, kk - row0 - slice * ATT_SUBTILE));

      if (!wait_or_abort(&full[s], (uint32_t)((it / nstage) & 1), abort_flag, p.s.dev_error)) break;
      if (nv > 0) {
        const uint32_t sbase =
            smem_addr(stage + (size_t)s * L.stage_bytes) + (uint32_t)(slice * ATT_SUBTILE * row_stride);
        // ---- S = Q K^T over the 16 rows (two n-tiles of 8 rows) ----
        float sc[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
          for (int kp = 0; kp < 4; ++kp) {
            // four 8x8 matrices: K rows 8j..8j+7, dims 32kp + 8*(lane/8) .. +7
            uint32_t b[4];
            const uint32_t addr = sbase + (uint32_t)((8 * j + (lane & 7)) * row_stride) +
                                  (uint32_t)((kvh * D + 32 * kp + 8 * (lane >> 3)) * 2);
            ldsm_x4(b, addr);
            mma_bf16(sc[j], qa[2 * kp], b[0], b[1]);
            mma_bf16(sc[j], qa[2 * kp + 1], b[2], b[3]);
          }
        }
        // ---- online softmax; rows >= nv are masked out ----
        float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool ok = 8 * j + 2 * tq + e < nv;
            sc[j][e] = ok ? sc[j][e] * sl2 : -INFINITY;
            sc[j][2 + e] = ok ? sc[j][2 + e] * sl2 : -INFINITY;
            mx_lo = fmaxf(mx_lo, sc[j][e]);
            mx_hi = fmaxf(mx_hi, sc[j][2 + e]);
          }
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(FULL_MASK, mx_lo, 1));
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(FULL_MASK, mx_lo, 2));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(FULL_MASK, mx_hi, 1));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(FULL_MASK, mx_hi, 2));
        const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
        // padded heads (>= G) see all-zero scores, never -inf: every m stays finite
        const float a_lo = exp2f(m_lo - mn_lo), a_hi = exp2f(m_hi - mn_hi);   // -inf - x -> 0
        m_lo = mn_lo;
        m_hi = mn_hi;
        uint32_t pa[4];
        float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float p0 = exp2f(sc[j][0] - mn_lo), p1 = exp2f(sc[j][1] - mn_lo);
          const float p2 = exp2f(sc[j][2] - mn_hi), p3 = exp2f(sc[j][3] - mn_hi);
          ps_lo += p0 + p1;
          ps_hi += p2 + p3;
          pa[2 * j + 0] = pack_bf16(p0, p1);
          pa[2 * j + 1] = pack_bf16(p2, p3);
        }
        l_lo = l_lo * a_lo + ps_lo;
        l_hi = l_hi * a_hi + ps_hi;
        if (__any_sync(FULL_MASK, a_lo != 1.f || a_hi != 1.f)) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            o[t][0] *= a_lo;
            o[t][1] *= a_lo;
            o[t][2] *= a_hi;
            o[t][3] *= a_hi;
          }
        }
        // ---- O += P V: 16 n-tiles of 8 dims, k = the 16 rows ----
        const uint32_t pfrag[4] = {pa[0], pa[1], pa[2], pa[3]};
#pragma unroll
        for (int tp = 0; tp < 8; ++tp) {
          // four 8x8 matrices: (rows 0-7 | 8-15) x (dims 16tp..+7 | 16tp+8..+15), transposed
          uint32_t b[4];
          const uint32_t addr = sbase + (uint32_t)(((lane & 7) + 8 * ((lane >> 3) & 1)) * row_stride) +
                                (uint32_t)((g.v_off + kvh * D + 16 * tp + 8 * (lane >> 4)) * 2);
          ldsm_x4_t(b, addr);
          mma_bf16(o[2 * tp], pfrag, b[0], b[1]);
          mma_bf16(o[2 * tp + 1], pfrag, b[2], b[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      s = (s + 1 == nstage) ? 0 : s + 1;
    }
    if (r >= 0 && !*abort_flag) flush(r);
  }

  __syncthreads();
  if (*abort_flag) {
    // drain copies that may still be in flight (bounded) before the stages go away
    if (tid == 0)
      for (int s2 = 0; s2 < nstage; ++s2) {
        (void)mbar_wait_bounded(&full[s2], 0);
        (void)mbar_wait_bounded(&full[s2], 1);
      }
    __syncthreads();
    return;
  }

  // ---- arrival counters: the last CTA of a request merges its partials ------------
  __threadfence();
  __syncthreads();
  int r_last = ri;
  while (prefix[r_last + 1] <= u1 - 1) ++r_last;
  for (int rr = ri; rr <= r_last; ++rr) {
    if (prefix[rr + 1] == prefix[rr]) continue;   // request without units
    if (tid == 0) {
      const int c_first = owner_of(prefix[rr], U, Gc);
      const int c_last = owner_of(prefix[rr + 1] - 1, U, Gc);
      const unsigned prev = atomicAdd(&p.s.att_counter[rr], 1u);
      s_last[0] = prev == (unsigned)(c_last - c_first);
      s_last[1] = c_last - c_first + 1;
    }
    __syncthreads();
    if (s_last[0]) {
      __threadfence();
      const int nparts = s_last[1] * NSLICE;
      const float* po = p.s.part_o + (long long)rr * p.att_parts * HQ * D;
      const float* pml = p.s.part_ml + (long long)rr * p.att_parts * HQ * 2;
      uint16_t* out = p.out + (long long)rr * HQ * D;
      for (int e = tid; e < HQ * D; e += THREADS) {
        const int h = e / D;
        float M = -INFINITY;
        for (int q = 0; q < nparts; ++q) M = fmaxf(M, __ldcg(pml + ((long long)q * HQ + h) * 2));
        float Ls = 0.f, O = 0.f;
        for (int q = 0; q < nparts; ++q) {
          const float mq = __ldcg(pml + ((long long)q * HQ + h) * 2);
          const float w = exp2f(mq - M);
          Ls = fmaf(__ldcg(pml + ((long long)q * HQ + h) * 2 + 1), w, Ls);
          O = fmaf(__ldcg(po + (long long)q * HQ * D + e), w, O);
        }
        out[e] = __bfloat16_as_ushort(__float2bfloat16_rn(O / Ls));
      }
      if (tid == 0) p.s.att_counter[rr] = 0;
    }
    __syncthreads();
  }
}

template <int G, int HKV>
static cudaError_t run_gqa(const DecodeParams* p, size_t smem, cudaStream_t st) {
  auto kern = attn_gqa_kernel<G, HKV>;
  if (p == nullptr)   // prepare: allow the shared memory this shape needs
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  kern<<<p->att_grid, THREADS, smem, st>>>(*p, attention_stages(p->g, smem));
  return cudaGetLastError();
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

cudaError_t prepare_attention(const Geometry& g, size_t smem) { return dispatch(g, nullptr, smem, 0); }

cudaError_t launch_attention(const DecodeParams& p, size_t smem, cudaStream_t st) {
  return dispatch(p.g, &p, smem, st);
}

}  // namespace hs
