// Append path (one new token per step, or a bulk prefill): index keys to the
// HBM key store, K/V rows to the authoritative copy in pinned host memory, and
// the request's length advanced once every CTA of the request has read it.
//
// Method: "KV卸载上主机:HiSparse、PDD与DDR4回收", section "论文1：HiSparse" —
// host DRAM holds the complete, authoritative KV of every active request, so
// each new token's K/V goes there; the hot cache is only filled by RESOLVE.
#include "hs_internal.cuh"

namespace hs {

// grid (ceil(n_tok / APP_TOKENS_PER_CTA), n_req); block APP_THREADS
__global__ void __launch_bounds__(APP_THREADS) append_kernel(AppendParams p) {
  const Geometry& g = p.g;
  const int ri = blockIdx.y;
  const int req = p.req_ids ? p.req_ids[ri] : ri;
  if (req < 0 || req >= g.max_requests) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(p.s.dev_error, HS_DEVERR_REQ_RANGE);
    return;
  }
  const long long rl = (long long)req * g.n_layers + p.layer;
  __shared__ int s_len;
  if (threadIdx.x == 0) s_len = p.s.length[rl];
  __syncthreads();
  const int len = s_len;
  const bool fits = (long long)len + p.n_tok <= g.max_context;

  if (fits) {
    const int t0 = blockIdx.x * APP_TOKENS_PER_CTA;
    const int nt = min(APP_TOKENS_PER_CTA, p.n_tok - t0);
    // index keys: d_idx bytes per token, 16-byte vectors
    const int kvec = g.d_idx / 16;
    const int4* ksrc = reinterpret_cast<const int4*>(p.keys + ((long long)ri * p.n_tok + t0) * g.d_idx);
    int4* kdst = reinterpret_cast<int4*>(p.s.idx_keys + (rl * g.max_context + len + t0) * g.d_idx);
    for (int e = threadIdx.x; e < nt * kvec; e += APP_THREADS) kdst[e] = ksrc[e];
    // K/V rows -> pinned host store (writes cross the host link)
    const int rvec = g.row_bytes / 16;
    const int4* rsrc = reinterpret_cast<const int4*>(p.kv_rows + ((long long)ri * p.n_tok + t0) * g.row_elems);
    int4* rdst = reinterpret_cast<int4*>(p.s.host_kv + (rl * g.max_context + len + t0) * g.row_elems);
    const int total = nt * rvec;
    for (int e = threadIdx.x; e < total; e += 4 * APP_THREADS) {
      int4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e + u * APP_THREADS < total) v[u] = rsrc[e + u * APP_THREADS];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e + u * APP_THREADS < total) rdst[e + u * APP_THREADS] = v[u];
    }
    // page mode: a page can be resident before all of its positions exist; the
    // rows appended to a resident page go to its slot as well (write-through)
    if (g.page_shift > 0) {
      const int psh = g.page_shift;
      const int32_t* ptab = p.s.page + rl * g.max_context;
      unsigned char* hot = reinterpret_cast<unsigned char*>(p.s.hot) + (size_t)rl * g.hot_slots * g.row_bytes;
      for (int i = 0; i < nt; ++i) {
        const int pos = len + t0 + i;
        const int ps = ptab[pos >> psh];
        if (ps < 0 || ps >= (g.hot_slots >> psh)) continue;
        int4* hdst = reinterpret_cast<int4*>(hot + (size_t)((ps << psh) + (pos & ((1 << psh) - 1))) * g.row_bytes);
        for (int e = threadIdx.x; e < rvec; e += APP_THREADS) hdst[e] = rsrc[i * rvec + e];
      }
    }
  }

  if (gridDim.x == 1) {   // one CTA per request (decode-time appends): no arrival counter
    __syncthreads();
    if (threadIdx.x == 0) {
      if (fits) {
        p.s.length[rl] = len + p.n_tok;
        atomicAdd(&p.s.glob[1], (unsigned long long)p.n_tok * g.row_bytes);
      } else {
        set_error(p.s.dev_error, HS_DEVERR_CAPACITY);
      }
    }
    return;
  }
  // The last CTA of this request (all others have read `len` by then) advances
  // the length and resets the arrival counter for the next call.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&p.s.app_counter[req], 1u);
    if (prev == gridDim.x - 1) {
      p.s.app_counter[req] = 0;
      if (fits) {
        p.s.length[rl] = len + p.n_tok;
        atomicAdd(&p.s.glob[1], (unsigned long long)p.n_tok * g.row_bytes);
      } else {
        set_error(p.s.dev_error, HS_DEVERR_CAPACITY);
      }
    }
  }
}

// Page mode: the element-wise maximum and minimum of the index keys of every page
// an append touched, recomputed whole from the key store: pages
// (len - n_tok) / P .. (len - 1) / P of the length after the append (the same
// pages again when the append was rejected, which rewrites the same values).
// grid (x, n_req); block APP_THREADS; one thread per 16-byte column chunk of a page
__global__ void __launch_bounds__(APP_THREADS) page_bound_kernel(AppendParams p) {
  const Geometry& g = p.g;
  const int ri = blockIdx.y;
  const int req = p.req_ids ? p.req_ids[ri] : ri;
  if (req < 0 || req >= g.max_requests) return;
  const long long rl = (long long)req * g.n_layers + p.layer;
  const int len = p.s.length[rl];
  if (len <= 0) return;
  const int psh = g.page_shift, P = 1 << psh;
  const int lo = max(0, len - p.n_tok) >> psh, hi = (len - 1) >> psh;
  const int hc = g.d_idx / 16;
  const int total = (hi - lo + 1) * hc;
  const int8_t* keys = p.s.idx_keys + rl * g.max_context * g.d_idx;
  int8_t* bound = p.s.pbound + rl * (long long)g.max_pages * 2 * g.d_idx;
  for (int e = blockIdx.x * APP_THREADS + threadIdx.x; e < total; e += gridDim.x * APP_THREADS) {
    const int pg = lo + e / hc, c = e % hc;
    const int r0 = pg << psh, r1 = min(len, r0 + P);
    int4 mx = *reinterpret_cast<const int4*>(keys + (long long)r0 * g.d_idx + c * 16);
    int4 mn = mx;
    for (int r = r0 + 1; r < r1; ++r) {
      const int4 v = *reinterpret_cast<const int4*>(keys + (long long)r * g.d_idx + c * 16);
      mx = vmax16(mx, v);
      mn = vmin16(mn, v);
    }
    int4* dst = reinterpret_cast<int4*>(bound + (long long)pg * 2 * g.d_idx);
    dst[c] = mx;
    dst[hc + c] = mn;
  }
}

__global__ void init_order_kernel(int32_t* order, long long n_lists, int B) {
  const long long total = n_lists * B;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x)
    order[i] = (int32_t)(i % B);
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t st) {
  dim3 grid((p.n_tok + APP_TOKENS_PER_CTA - 1) / APP_TOKENS_PER_CTA, p.n_req);
  append_kernel<<<grid, APP_THREADS, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_page_bounds(const AppendParams& p, cudaStream_t st) {
  const int pages = (p.n_tok >> p.g.page_shift) + 2;   // the most pages an append of n_tok touches
  const int work = pages * (p.g.d_idx / 16);
  dim3 grid(std::min((work + APP_THREADS - 1) / APP_THREADS, 1024), p.n_req);
  page_bound_kernel<<<grid, APP_THREADS, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_init_order(int32_t* order, long long n_lists, int B, cudaStream_t st) {
  const long long total = n_lists * B;
  int blocks = (int)std::min<long long>((total + 255) / 256, 4096);
  if (blocks < 1) blocks = 1;
  init_order_kernel<<<blocks, 256, 0, st>>>(order, n_lists, B);
  return cudaGetLastError();
}

}  // namespace hs
