// Sparse attention over a shared latent row (MLA-style cache): every selected
// position holds one latent vector of 576 bf16, read as K (all 576 dims) and as
// V (its first 512 dims) by every query head; 16 to 128 query heads.
//
// Method: "Heterogeneous LLM Serving with General-Purpose Processing-Near-Memory
// for Retrieval-Based Sparse Attention" (vsvnakers.github.io), "核心公式与算法",
// formula 2: softmax over the selected positions only.  "KV卸载上主机:
// HiSparse、PDD与DDR4回收", "论文1：HiSparse": only where rows live changes, so
// the result must not depend on B.
//
// Design (sm_103a).  With 128 heads sharing each 1152-byte row the kernel does
// ~240 flop per byte, so the products run on the tensor cores (mma.sync
// m16n8k16, bf16 in, fp32 accumulate):
//  * Work items are (request, group of 16*NMT heads, unit of 64/NMT selected
//    rows), flattened in that order and split into equal contiguous ranges, one
//    per CTA (persistent, one CTA per SM).  The split depends only on k_eff and
//    the grid, never on B.  With NMT = 2 (32 heads x 32 rows) an item moves half
//    the bytes of a 64-row item for the same tensor work, so four stages fit in
//    shared memory; rows are re-read once per head group, from L2.
//  * Warp 8 (stager) copies an item's rows from their hot slots into shared
//    memory with 1-D bulk async copies (cp.async.bulk, mbarrier completion).
//    RESOLVE has already pulled every missed row into its slot (latent rows are
//    shared by all head groups, so they cross the host link once).
//  * Warps 0-7: S = Q K^T with warp w taking head tile w / (8/NMT) and row tile
//    w % (8/NMT) (36 k-steps over the 576 dims in four independent accumulator
//    chains; Q of the head group in shared memory); per-head maxima and sums of
//    the item's rows are exchanged through shared memory; P goes to shared memory
//    as bf16; then warp w accumulates O[all heads of the item, dims 64w..64w+63]
//    += P V (V fragments by ldmatrix.trans).  Online softmax in fp32 with exp2;
//    rows past k_eff are masked and zero-filled.
//  * Each (CTA, request, head group) writes a partial (m, l, o); the merge kernel
//    combines them in part order.
#include <cuda_bf16.h>

#include "hs_internal.cuh"

namespace hs {

namespace {

constexpr int MLA_DK = 576, MLA_DV = 512;
constexpr int MLA_NCONS = 8;                      // consumer warps
constexpr int MLA_STAGER = MLA_NCONS;             // warp index of the stager
constexpr int MLA_THREADS = (MLA_NCONS + 1) * 32;
constexpr int MLA_ROW_STRIDE = MLA_DK * 2 + 16;   // shared-memory row pitch (bank spread for ldmatrix)
constexpr int MLA_MAX_STAGES = 4;
constexpr size_t MLA_SMEM_LIMIT = 227 * 1024;

// 16-head tiles per item: two (32 heads x 32 rows) when the heads allow it
__host__ __device__ inline int mla_nmt(const Geometry& g) { return g.h_q >= 32 ? 2 : 1; }
__host__ __device__ inline int mla_rows(const Geometry& g) { return 64 / mla_nmt(g); }

__host__ __device__ inline size_t mla_align(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct MlaLayout {
  size_t bar, prefix, q, p, red, stage, stage_bytes, total;
  int nstage;
};

__host__ __device__ inline MlaLayout mla_layout(const Geometry& g) {
  const int nmt = mla_nmt(g), rows = mla_rows(g);
  MlaLayout L;
  size_t off = 0;
  L.bar = off;
  off += 8 * 2 * MLA_MAX_STAGES + 16;   // full/empty barriers, abort flag
  off = mla_align(off, 128);
  L.prefix = off;   // first item, k_eff and request id of each request
  off += mla_align((size_t)(g.max_requests + 1) * 4 * 3, 128);
  L.q = off;        // Q of the item's heads
  off += (size_t)16 * nmt * MLA_ROW_STRIDE;
  L.p = off;        // P [heads][rows] bf16
  off += (size_t)16 * nmt * (rows * 2 + 16);
  L.red = off;      // per (head tile, row tile) head maxima (two buffers) and sums
  off += (size_t)3 * 8 * 16 * 4;
  off = mla_align(off, 128);
  L.stage = off;
  L.stage_bytes = (size_t)rows * MLA_ROW_STRIDE;
  int ns = MLA_MAX_STAGES;
  while (ns > 2 && off + ns * L.stage_bytes > MLA_SMEM_LIMIT) --ns;
  L.nstage = ns;
  off += (size_t)ns * L.stage_bytes;
  L.total = off;
  return L;
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barrier of the 256 consumer threads that also ORs a flag over them.
__device__ __forceinline__ bool consumers_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 256, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ bool wait_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
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

__device__ __forceinline__ int owner(long long u, long long U, int G) {
  return (int)(((u + 1) * G + U - 1) / U) - 1;
}

}  // namespace

int mla_parts(const Geometry& g) { return (g.top_k + mla_rows(g) - 1) / mla_rows(g) + 1; }
size_t mla_smem_bytes(const Geometry& g) { return mla_layout(g).total; }

template <int HQ, int NMT>
__global__ void __launch_bounds__(MLA_THREADS, 1) attn_mla_kernel(DecodeParams p) {
  constexpr int GH = 16 * NMT;          // heads per item
  constexpr int ROWS = 64 / NMT;        // rows per item
  constexpr int NT = ROWS / 8;          // row tiles (mma N) per item
  constexpr int NHG = HQ / GH;
  constexpr int P_STRIDE = ROWS * 2 + 16;
  const Geometry& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = g.top_k;
  const int c = blockIdx.x;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  const MlaLayout L = mla_layout(g);
  const int nstage = L.nstage;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + L.bar);
  uint64_t* empty = full + MLA_MAX_STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + MLA_MAX_STAGES);
  int* prefix = reinterpret_cast<int*>(smem_raw + L.prefix);
  int* kk_s = prefix + (g.max_requests + 1);
  int* req_s = kk_s + (g.max_requests + 1);
  unsigned char* qs = smem_raw + L.q;
  unsigned char* ps = smem_raw + L.p;
  float* smax = reinterpret_cast<float*>(smem_raw + L.red);   // [2][8 blocks][16]
  float* ssum = smax + 2 * 8 * 16;                            // [8 blocks][16]
  unsigned char* stage = smem_raw + L.stage;
  __shared__ int scan_tmp[MLA_THREADS / 32 + 1];
  HS_TRACE(p, 2, 0);

  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MLA_NCONS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  griddep_wait();   // selection, slots (rows pulled by RESOLVE), lengths, q
  griddep_launch_dependents();

  // ---- work list: NHG * ceil(k_eff / ROWS) items per request ----
  int carry = 0;
  for (int base = 0; base < p.n_req; base += MLA_THREADS) {
    const int i = base + tid;
    int items = 0;
    if (i < p.n_req) {
      const int req = p.req_ids ? p.req_ids[i] : i;
      int kk = 0;
      if (req >= 0 && req < g.max_requests) kk = min(K, p.s.length[(long long)req * g.n_layers + p.layer]);
      items = NHG * ((kk + ROWS - 1) / ROWS);
      kk_s[i] = kk;
      req_s[i] = req;
      if (kk == 0 && i % (int)gridDim.x == c) {   // nothing selected: the output is defined as 0
        uint16_t* out = p.out + (long long)i * HQ * MLA_DV;
        for (int e = 0; e < HQ * MLA_DV; ++e) out[e] = 0;
        if (req >= 0 && req < g.max_requests) set_error(p.s.dev_error, HS_DEVERR_EMPTY);
      }
    }
    int tot;
    const int ex = block_exclusive_scan<MLA_THREADS>(items, scan_tmp, &tot);
    if (i < p.n_req) prefix[i] = carry + ex;
    carry += tot;
  }
  if (tid == 0) prefix[p.n_req] = carry;
  __syncthreads();
  const long long U = carry;
  const int Gc = (int)max(1LL, min((long long)gridDim.x, U));
  if (c == 0)   // partials of each (request, head group), for the merge kernel
    for (int e = tid; e < p.n_req * NHG; e += MLA_THREADS) {
      const int i = e / NHG, hg = e % NHG;
      const int ui = (kk_s[i] + ROWS - 1) / ROWS;
      const long long f0 = prefix[i] + (long long)hg * ui;
      p.s.att_nparts[(long long)i * NHG + hg] = ui ? owner(f0 + ui - 1, U, Gc) - owner(f0, U, Gc) + 1 : 0;
    }
  if (U == 0 || c >= Gc) return;
  const long long u0 = (long long)c * U / Gc, u1 = (long long)(c + 1) * U / Gc;
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
  struct Item {
    int r, hg, unit, nv;
  };
  auto decode = [&](long long f, int& r) -> Item {
    while (prefix[r + 1] <= f) ++r;
    Item it;
    it.r = r;
    const int ui = (kk_s[r] + ROWS - 1) / ROWS;
    const int local = (int)(f - prefix[r]);
    it.hg = local / ui;
    it.unit = local - it.hg * ui;
    it.nv = min(ROWS, kk_s[r] - it.unit * ROWS);
    return it;
  };

  if (warp == MLA_STAGER) {
    // ============================ stager warp ============================
    int r = ri;
    int s = 0;
    long long it = 0;
    for (long long f = u0; f < u1; ++f, ++it) {
      const Item w = decode(f, r);
      const long long rl = (long long)req_s[w.r] * g.n_layers + p.layer;
      int slot[(ROWS + 31) / 32];
#pragma unroll
      for (int h = 0; h < (ROWS + 31) / 32; ++h) {
        const int j = lane + 32 * h;
        slot[h] = j < w.nv ? p.s.slot_of_sel[(long long)w.r * K + w.unit * ROWS + j] : 0;
      }
      if (it >= nstage &&
          !__all_sync(FULL_MASK, wait_abort(&empty[s], (uint32_t)(((it / nstage) + 1) & 1), abort_flag,
                                            p.s.dev_error)))
        break;
      unsigned char* st_s = stage + (size_t)s * L.stage_bytes;
      if (w.nv < ROWS) {   // rows past k_eff: zeros keep the masked products finite
        const int rvec = MLA_DK * 2 / 16;
        for (int e = lane; e < (ROWS - w.nv) * rvec; e += 32) {
          const int j = w.nv + e / rvec;
          *reinterpret_cast<int4*>(st_s + (size_t)j * MLA_ROW_STRIDE + (e % rvec) * 16) = make_int4(0, 0, 0, 0);
        }
      }
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&full[s], (uint32_t)(w.nv * g.row_bytes));
      }
      __syncwarp();
      const unsigned char* hot =
          reinterpret_cast<const unsigned char*>(p.s.hot) + (size_t)rl * g.hot_slots * g.row_bytes;
#pragma unroll
      for (int h = 0; h < (ROWS + 31) / 32; ++h) {
        const int j = lane + 32 * h;
        if (j < w.nv) {
          int sl = slot[h];
          if (sl < 0 || sl >= g.hot_slots) {   // never expected (RESOLVE fills every slot): stay in bounds
            set_error(p.s.dev_error, HS_DEVERR_METADATA);
            sl = 0;
          }
          bulk_g2s(st_s + (size_t)j * MLA_ROW_STRIDE, hot + (size_t)sl * g.row_bytes, (uint32_t)g.row_bytes,
                   &full[s]);
        }
      }
      s = (s + 1 == nstage) ? 0 : s + 1;
    }
  } else {
    // ============================ consumer warps ============================
    const int gq = lane >> 2, tq = lane & 3;
    const int smt = warp / NT, snt = warp % NT;   // this warp's (head tile, row tile) of S
    const float sl2 = p.scale_log2;
    const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1);   // ldmatrix row of this lane (16-row operands)
    const int lcol = 8 * (lane >> 4);                        // and its column offset
    float o[NMT][8][4];
    float m[NMT][2], l[NMT][2];   // heads 16 mt + gq and 16 mt + gq + 8
    int cur_r = -1, cur_hg = -1;
    int r = ri;
    int s = 0;
    long long it = 0;

    auto flush = [&](int rq, int hg) {
      const long long f0 = prefix[rq] + (long long)hg * ((kk_s[rq] + ROWS - 1) / ROWS);
      const int part = c - owner(f0, U, Gc);
      const long long base = ((long long)rq * p.att_parts + part) * HQ + hg * GH;
      float* po = p.s.part_o + base * MLA_DV;
      float* pml = p.s.part_ml + base * 2;
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int d = 64 * warp + 8 * t + 2 * tq;
          *reinterpret_cast<float2*>(po + (long long)(16 * mt + gq) * MLA_DV + d) = make_float2(o[mt][t][0], o[mt][t][1]);
          *reinterpret_cast<float2*>(po + (long long)(16 * mt + gq + 8) * MLA_DV + d) =
              make_float2(o[mt][t][2], o[mt][t][3]);
        }
        if (warp == 0 && tq == 0) {
          *reinterpret_cast<float2*>(pml + (16 * mt + gq) * 2) = make_float2(m[mt][0], l[mt][0]);
          *reinterpret_cast<float2*>(pml + (16 * mt + gq + 8) * 2) = make_float2(m[mt][1], l[mt][1]);
        }
      }
    };

    for (long long f = u0; f < u1; ++f, ++it) {
      const Item w = decode(f, r);
      if (w.r != cur_r || w.hg != cur_hg) {
        if (cur_r >= 0) flush(cur_r, cur_hg);
        cur_r = w.r;
        cur_hg = w.hg;
        consumers_sync();   // every warp is done with the previous group's Q
        const int4* qsrc = reinterpret_cast<const int4*>(p.q + ((long long)w.r * HQ + w.hg * GH) * MLA_DK);
        for (int e = tid; e < GH * MLA_DK / 8; e += MLA_NCONS * 32) {
          const int h = e / (MLA_DK / 8), v = e % (MLA_DK / 8);
          *reinterpret_cast<int4*>(qs + (size_t)h * MLA_ROW_STRIDE + v * 16) = qsrc[e];
        }
        consumers_sync();
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll
          for (int t = 0; t < 8; ++t) o[mt][t][0] = o[mt][t][1] = o[mt][t][2] = o[mt][t][3] = 0.f;
          m[mt][0] = m[mt][1] = -INFINITY;
          l[mt][0] = l[mt][1] = 0.f;
        }
      }
      const bool ok = wait_abort(&full[s], (uint32_t)((it / nstage) & 1), abort_flag, p.s.dev_error);
      const unsigned char* st_s = stage + (size_t)s * L.stage_bytes;
      // ---- S = Q K^T for head tile smt x row tile snt ----
      float sc[4];
      {
        float acc[4][4] = {};
        const uint32_t rowa = smem_addr(st_s + (size_t)(8 * snt + (lane & 7)) * MLA_ROW_STRIDE) + 16 * (lane >> 3);
        const uint32_t qa = smem_addr(qs + (size_t)(16 * smt + lrow) * MLA_ROW_STRIDE) + 2 * lcol;
#pragma unroll
        for (int kp2 = 0; kp2 < MLA_DK / 64; ++kp2) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int kp = 2 * kp2 + h2;
            uint32_t b[4], a0[4], a1[4];
            ldsm4(b, rowa + 64 * kp);          // K rows x dims 32kp .. 32kp+31
            ldsm4(a0, qa + 64 * kp);           // Q dims 32kp .. +15
            ldsm4(a1, qa + 64 * kp + 32);      // Q dims 32kp+16 .. +31
            mma16816(acc[2 * h2], a0, b[0], b[1]);
            mma16816(acc[2 * h2 + 1], a1, b[2], b[3]);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
      }
      // ---- block maxima per head ----
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool okr = 8 * snt + 2 * tq + e < w.nv;
        sc[e] = okr ? sc[e] * sl2 : -INFINITY;
        sc[2 + e] = okr ? sc[2 + e] * sl2 : -INFINITY;
        mx_lo = fmaxf(mx_lo, sc[e]);
        mx_hi = fmaxf(mx_hi, sc[2 + e]);
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(FULL_MASK, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(FULL_MASK, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(FULL_MASK, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(FULL_MASK, mx_hi, 2));
      float* smx = smax + (it & 1) * 8 * 16;   // [block = warp][16 heads of its tile]
      if (tq == 0) {
        smx[warp * 16 + gq] = mx_lo;
        smx[warp * 16 + gq + 8] = mx_hi;
      }
      if (consumers_sync_or(!ok)) break;   // all consumer warps leave together
      // new running maxima of every head this lane covers (all head tiles), from
      // the blocks of each head tile (same order in every warp)
      float mnew[NMT][2], alpha[NMT][2];
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
        float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
        for (int q = 0; q < NT; ++q) {
          t0 = fmaxf(t0, smx[(mt * NT + q) * 16 + gq]);
          t1 = fmaxf(t1, smx[(mt * NT + q) * 16 + gq + 8]);
        }
        mnew[mt][0] = fmaxf(m[mt][0], t0);   // finite: every item has a valid row
        mnew[mt][1] = fmaxf(m[mt][1], t1);
        alpha[mt][0] = exp2f(m[mt][0] - mnew[mt][0]);
        alpha[mt][1] = exp2f(m[mt][1] - mnew[mt][1]);
      }
      // P of this warp's block, and its per-head sums
      {
        const float ml = mnew[smt][0], mh = mnew[smt][1];
        const float p0 = exp2f(sc[0] - ml), p1 = exp2f(sc[1] - ml);
        const float p2 = exp2f(sc[2] - mh), p3 = exp2f(sc[3] - mh);
        *reinterpret_cast<uint32_t*>(ps + (size_t)(16 * smt + gq) * P_STRIDE + 2 * (8 * snt + 2 * tq)) =
            pack2_bf16(p0, p1);
        *reinterpret_cast<uint32_t*>(ps + (size_t)(16 * smt + gq + 8) * P_STRIDE + 2 * (8 * snt + 2 * tq)) =
            pack2_bf16(p2, p3);
        float su_lo = p0 + p1, su_hi = p2 + p3;
        su_lo += __shfl_xor_sync(FULL_MASK, su_lo, 1);
        su_lo += __shfl_xor_sync(FULL_MASK, su_lo, 2);
        su_hi += __shfl_xor_sync(FULL_MASK, su_hi, 1);
        su_hi += __shfl_xor_sync(FULL_MASK, su_hi, 2);
        if (tq == 0) {
          ssum[warp * 16 + gq] = su_lo;
          ssum[warp * 16 + gq + 8] = su_hi;
        }
      }
      consumers_sync();
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
        float ts0 = 0.f, ts1 = 0.f;
#pragma unroll
        for (int q = 0; q < NT; ++q) {   // fixed order: every warp gets the same l
          ts0 += ssum[(mt * NT + q) * 16 + gq];
          ts1 += ssum[(mt * NT + q) * 16 + gq + 8];
        }
        l[mt][0] = l[mt][0] * alpha[mt][0] + ts0;
        l[mt][1] = l[mt][1] * alpha[mt][1] + ts1;
        m[mt][0] = mnew[mt][0];
        m[mt][1] = mnew[mt][1];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          o[mt][t][0] *= alpha[mt][0];
          o[mt][t][1] *= alpha[mt][0];
          o[mt][t][2] *= alpha[mt][1];
          o[mt][t][3] *= alpha[mt][1];
        }
      }
      // ---- O[:, 64*warp .. +63] += P V over the item's rows ----
      {
        const uint32_t pa_base = smem_addr(ps + (size_t)lrow * P_STRIDE) + 2 * lcol;
        const uint32_t v_base = smem_addr(st_s + (size_t)lrow * MLA_ROW_STRIDE) + 2 * (64 * warp + lcol);
#pragma unroll
        for (int ks = 0; ks < ROWS / 16; ++ks) {
          uint32_t pa[NMT][4];
#pragma unroll
          for (int mt = 0; mt < NMT; ++mt)
            ldsm4(pa[mt], pa_base + (uint32_t)(16 * mt * P_STRIDE) + 32 * ks);   // P heads 16mt.. x rows 16ks..
#pragma unroll
          for (int tp = 0; tp < 4; ++tp) {
            uint32_t b[4];
            ldsm4_t(b, v_base + (uint32_t)(16 * ks * MLA_ROW_STRIDE) + 32 * tp);
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt) {
              mma16816(o[mt][2 * tp], pa[mt], b[0], b[1]);
              mma16816(o[mt][2 * tp + 1], pa[mt], b[2], b[3]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive1(&empty[s]);
      s = (s + 1 == nstage) ? 0 : s + 1;
    }
    if (cur_r >= 0 && !*abort_flag) flush(cur_r, cur_hg);
  }
  __syncthreads();
  if (*abort_flag && tid == 0)   // drain copies that may still be in flight (bounded)
    for (int s2 = 0; s2 < nstage; ++s2) {
      (void)mbar_wait_bounded(&full[s2], 0);
      (void)mbar_wait_bounded(&full[s2], 1);
    }
  HS_TRACE(p, 2, 14);
}

template <int HQ>
static cudaError_t run_mla(const DecodeParams* p, size_t smem, cudaStream_t st) {
  constexpr int NMT = HQ >= 32 ? 2 : 1;
  auto kern = attn_mla_kernel<HQ, NMT>;
  if (p == nullptr) return allow_smem(kern, smem);
  cudaError_t e = launch_pdl(kern, dim3(p->att_grid), dim3(MLA_THREADS), smem, st, *p);
  if (e != cudaSuccess) return e;
  return launch_merge(*p, st);
}

cudaError_t dispatch_mla(const Geometry& g, const DecodeParams* p, size_t smem, cudaStream_t st) {
  switch (g.h_q) {
    case 16: return run_mla<16>(p, smem, st);
    case 32: return run_mla<32>(p, smem, st);
    case 64: return run_mla<64>(p, smem, st);
    case 128: return run_mla<128>(p, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hs
