// Sparse attention over the selected rows (GQA, head dim 128), split over the
// selection, with the split results merged by the last CTA of each request.
//
// Method: "Heterogeneous LLM Serving with General-Purpose Processing-Near-Memory
// for Retrieval-Based Sparse Attention" (vsvnakers.github.io), "核心公式与算法",
// formula 2: softmax(Q K^T / sqrt(d_k), masked to the retrieved entries) V —
// read as a softmax over the selected positions only.  "KV卸载上主机:
// HiSparse、PDD与DDR4回收", "论文1：HiSparse": the attention math is unchanged
// by the cache, so the result must not depend on where the rows sit.
//
// Design (sm_103a), HBM-bound (about 4 flop per byte for 4 q heads per kv head),
// so CUDA cores, not tensor cores:
//  * grid (splits, requests); a CTA owns ATT_SPLIT consecutive selection
//    ordinals, so the work split depends only on k_eff, never on B or on slots;
//  * each selected row (all kv heads, contiguous in its hot slot) is copied
//    HBM -> shared memory by one 1-D bulk async copy into a row-padded layout
//    (16 extra bytes per row spread rows over all banks), two stages deep;
//  * warp w serves kv head w % H_kv and rows of slice w / H_kv of each tile;
//    scores: lane = (half of the head dim, row), q pre-scaled by scale*log2(e)
//    in fp32 shared memory; online softmax in fp32 (exp2); P.V: lane = 4 dims;
//  * partial (m, l, o) per (split, slice) in scratch; the last CTA of the
//    request (arrival counter) merges them in a fixed order and writes bf16.
// Rows are visited in ascending selection order and the merge order is fixed,
// so the output is bit-identical for any B and any slot placement.
#include <cuda_bf16.h>

#include "hs_internal.cuh"

namespace hs {

namespace {

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct AttLayout {
  size_t bar, qs, pbuf, stage, stage_bytes, total;
};

__host__ __device__ inline AttLayout att_layout(const Geometry& g, int G) {
  AttLayout L;
  const int nslice = ATT_WARPS / g.h_kv;
  const int tile = ATT_SUBTILE * nslice;
  const size_t row_stride = (size_t)g.row_bytes + ATT_ROW_PAD;
  size_t off = 0;
  L.bar = off;
  off += 64;
  L.qs = off;
  off += (size_t)g.h_q * 128 * 4;
  L.pbuf = off;
  off += (size_t)ATT_WARPS * ATT_SUBTILE * G * 4;
  off = align_up(off, 128);
  L.stage = off;
  L.stage_bytes = align_up((size_t)tile * row_stride, 128);
  off += ATT_STAGES * L.stage_bytes;
  L.total = off;
  return L;
}

}  // namespace

int attention_parts(const Geometry& g) {
  const int nsplit = (g.top_k + ATT_SPLIT - 1) / ATT_SPLIT;
  return nsplit * (ATT_WARPS / g.h_kv);
}

size_t attention_smem_bytes(const Geometry& g) { return att_layout(g, g.h_q / g.h_kv).total; }

template <int G, int HKV>
__global__ void __launch_bounds__(ATT_THREADS, 1) attn_gqa_kernel(DecodeParams p) {
  constexpr int NSLICE = ATT_WARPS / HKV;
  constexpr int TILE = ATT_SUBTILE * NSLICE;
  constexpr int D = 128;
  const Geometry& g = p.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ri = blockIdx.y;
  const int split = blockIdx.x;
  const int K = g.top_k;
  const int HQ = HKV * G;
  uint16_t* out = p.out + (long long)ri * HQ * D;

  const int req = p.req_ids ? p.req_ids[ri] : ri;
  int kk = 0;
  long long rl = 0;
  if (req >= 0 && req < g.max_requests) {
    rl = (long long)req * g.n_layers + p.layer;
    kk = min(K, p.s.length[rl]);
  }
  if (kk == 0) {   // nothing selected: the output is defined as 0
    if (split == 0) {
      for (int e = tid; e < HQ * D; e += ATT_THREADS) out[e] = 0;
      if (tid == 0 && req >= 0 && req < g.max_requests) set_error(p.s.dev_error, HS_DEVERR_EMPTY);
    }
    return;
  }
  const int nsplit = (kk + ATT_SPLIT - 1) / ATT_SPLIT;
  if (split >= nsplit) return;
  const int r0 = split * ATT_SPLIT;
  const int nrows = min(kk, r0 + ATT_SPLIT) - r0;
  const int ntiles = (nrows + TILE - 1) / TILE;

  extern __shared__ __align__(128) unsigned char smem_raw[];
  const AttLayout L = att_layout(g, G);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + L.bar);
  float* qs = reinterpret_cast<float*>(smem_raw + L.qs);
  float* pbuf = reinterpret_cast<float*>(smem_raw + L.pbuf);
  unsigned char* stage = smem_raw + L.stage;
  const int row_stride = g.row_bytes + ATT_ROW_PAD;

  // q (bf16) -> fp32 * scale * log2(e)
  const uint16_t* qg = p.q + (long long)ri * HQ * D;
  for (int e = tid; e < HQ * D; e += ATT_THREADS) qs[e] = __uint_as_float((uint32_t)qg[e] << 16) * p.scale_log2;
  if (tid == 0) {
    for (int s = 0; s < ATT_STAGES; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int32_t* sos = p.s.slot_of_sel + (long long)ri * K + r0;
  const unsigned char* hot = reinterpret_cast<const unsigned char*>(p.s.hot) + (size_t)rl * g.hot_slots * g.row_bytes;
  auto issue = [&](int t) {   // called by all lanes of warp 0
    const int s = t % ATT_STAGES;
    const int nr = min(TILE, nrows - t * TILE);
    if (lane == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bar[s], (uint32_t)(nr * g.row_bytes));
    }
    __syncwarp();
    for (int i = lane; i < nr; i += 32) {
      int slot = sos[t * TILE + i];
      if (slot < 0 || slot >= g.hot_slots) {   // never expected: keep the copy in bounds
        set_error(p.s.dev_error, HS_DEVERR_METADATA);
        slot = 0;
      }
      bulk_g2s(stage + s * L.stage_bytes + (size_t)i * row_stride, hot + (size_t)slot * g.row_bytes,
               (uint32_t)g.row_bytes, &bar[s]);
    }
  };
  if (warp == 0)
    for (int t = 0; t < ATT_STAGES && t < ntiles; ++t) issue(t);

  const int kvh = warp % HKV;
  const int slice = warp / HKV;
  const int half = lane >> 4, rrow = lane & 15;
  float m_run[G], l_run[G], o[G][4];
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    m_run[gg] = -INFINITY;
    l_run[gg] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) o[gg][c] = 0.f;
  }
  float* pw = pbuf + warp * ATT_SUBTILE * G;

  bool timed_out = false;
  int consumed = 0;
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % ATT_STAGES;
    const bool ok = mbar_wait_bounded(&bar[s], (uint32_t)((t / ATT_STAGES) & 1));
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    consumed = t + 1;
    const unsigned char* st = stage + s * L.stage_bytes;
    const int wr0 = slice * ATT_SUBTILE;
    const int nv = max(0, min(ATT_SUBTILE, nrows - t * TILE - wr0));
    if (nv > 0) {
      // ---- scores of the warp's 16 rows for its G heads --------------------
      float acc[G];
#pragma unroll
      for (int gg = 0; gg < G; ++gg) acc[gg] = 0.f;
      const unsigned char* krow = st + (size_t)(wr0 + rrow) * row_stride + (size_t)(kvh * D + half * 64) * 2;
      const float* qh = qs + (kvh * G) * D + half * 64;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 kc = *reinterpret_cast<const uint4*>(krow + c * 16);
        float kf[8];
        kf[0] = bf16lo(kc.x); kf[1] = bf16hi(kc.x);
        kf[2] = bf16lo(kc.y); kf[3] = bf16hi(kc.y);
        kf[4] = bf16lo(kc.z); kf[5] = bf16hi(kc.z);
        kf[6] = bf16lo(kc.w); kf[7] = bf16hi(kc.w);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float4 qa = *reinterpret_cast<const float4*>(qh + gg * D + c * 8);
          const float4 qb = *reinterpret_cast<const float4*>(qh + gg * D + c * 8 + 4);
          float a = acc[gg];
          a = fmaf(qa.x, kf[0], a); a = fmaf(qa.y, kf[1], a);
          a = fmaf(qa.z, kf[2], a); a = fmaf(qa.w, kf[3], a);
          a = fmaf(qb.x, kf[4], a); a = fmaf(qb.y, kf[5], a);
          a = fmaf(qb.z, kf[6], a); a = fmaf(qb.w, kf[7], a);
          acc[gg] = a;
        }
      }
      const bool valid = rrow < nv;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        float sc = acc[gg] + __shfl_xor_sync(FULL_MASK, acc[gg], 16);
        sc = valid ? sc : -INFINITY;
        float mx = sc;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, off));
        const float mnew = fmaxf(m_run[gg], mx);
        const float alpha = exp2f(m_run[gg] - mnew);   // m_run = -inf -> 0
        const float pv = valid ? exp2f(sc - mnew) : 0.f;
        float ps = pv;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) ps += __shfl_xor_sync(FULL_MASK, ps, off);
        l_run[gg] = l_run[gg] * alpha + ps;
        m_run[gg] = mnew;
#pragma unroll
        for (int c = 0; c < 4; ++c) o[gg][c] *= alpha;
        if (half == 0) pw[rrow * G + gg] = pv;
      }
      __syncwarp();
      // ---- P . V: lane owns 4 consecutive dims of the head -------------------
      const unsigned char* vb = st + (size_t)wr0 * row_stride + (size_t)(g.v_off + kvh * D + lane * 4) * 2;
#pragma unroll 4
      for (int i = 0; i < nv; ++i) {
        const uint2 vv = *reinterpret_cast<const uint2*>(vb + (size_t)i * row_stride);
        const float v0 = bf16lo(vv.x), v1 = bf16hi(vv.x), v2 = bf16lo(vv.y), v3 = bf16hi(vv.y);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float pg = pw[i * G + gg];
          o[gg][0] = fmaf(pg, v0, o[gg][0]);
          o[gg][1] = fmaf(pg, v1, o[gg][1]);
          o[gg][2] = fmaf(pg, v2, o[gg][2]);
          o[gg][3] = fmaf(pg, v3, o[gg][3]);
        }
      }
      __syncwarp();
    }
    __syncthreads();   // stage s is free
    if (warp == 0 && t + ATT_STAGES < ntiles) issue(t + ATT_STAGES);
  }
  if (timed_out) {
    if (tid == 0) {
      const int issued = min(ntiles, consumed + ATT_STAGES);
      for (int t = consumed; t < issued; ++t)
        (void)mbar_wait_bounded(&bar[t % ATT_STAGES], (uint32_t)((t / ATT_STAGES) & 1));
      set_error(p.s.dev_error, HS_DEVERR_TIMEOUT);
    }
    __syncthreads();
  }

  // ---- partial results of this (split, slice) ----------------------------------
  const int parts = p.att_parts;
  const int part = split * NSLICE + slice;
  float* po = p.s.part_o + (long long)ri * parts * HQ * D;
  float* pml = p.s.part_ml + (long long)ri * parts * HQ * 2;
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    const int h = kvh * G + gg;
    *reinterpret_cast<float4*>(po + ((long long)part * HQ + h) * D + lane * 4) =
        make_float4(o[gg][0], o[gg][1], o[gg][2], o[gg][3]);
    if (lane == 0) {
      pml[((long long)part * HQ + h) * 2 + 0] = m_run[gg];
      pml[((long long)part * HQ + h) * 2 + 1] = l_run[gg];
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) {
    const unsigned prev = atomicAdd(&p.s.att_counter[ri], 1u);
    s_last = prev == (unsigned)(nsplit - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // ---- last CTA of the request: merge the parts in a fixed order -----------------
  const int nparts = nsplit * NSLICE;
  for (int e = tid; e < HQ * D; e += ATT_THREADS) {
    const int h = e / D;
    float M = -INFINITY;
    for (int q = 0; q < nparts; ++q) M = fmaxf(M, __ldcg(pml + ((long long)q * HQ + h) * 2));
    float Lsum = 0.f, O = 0.f;
    for (int q = 0; q < nparts; ++q) {
      const float mq = __ldcg(pml + ((long long)q * HQ + h) * 2);
      const float lq = __ldcg(pml + ((long long)q * HQ + h) * 2 + 1);
      const float w = exp2f(mq - M);
      Lsum = fmaf(lq, w, Lsum);
      O = fmaf(__ldcg(po + (long long)q * HQ * D + e), w, O);
    }
    const float r = O / Lsum;
    out[e] = __bfloat16_as_ushort(__float2bfloat16_rn(r));
  }
  if (tid == 0) p.s.att_counter[ri] = 0;
}

template <int G, int HKV>
static cudaError_t run_gqa(const DecodeParams* p, size_t smem, cudaStream_t st) {
  auto kern = attn_gqa_kernel<G, HKV>;
  if (p == nullptr)   // prepare: allow the shared memory this shape needs
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid((p->g.top_k + ATT_SPLIT - 1) / ATT_SPLIT, p->n_req);
  kern<<<grid, ATT_THREADS, smem, st>>>(*p);
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
