// hs_indexer_topk_static: indexer scores and exact top-k selection for callers
// that cannot allocate device memory — code running where cudaMalloc is not
// available or not allowed (inside another allocator's critical section, under a
// memory pool that forbids side allocations, in a plugin handed only raw
// pointers).  Its scratch lives in one file-scope device array; the caller passes
// inputs and outputs only.  See include/hs.h for the contract.
#include "hs_internal.cuh"

namespace hs {
namespace {
constexpr int ST_MAX_REQUESTS = 64;
constexpr long long ST_MAX_POSITIONS = 1ll << 21;   // sum over requests of n_max rounded up to 4
constexpr size_t ST_OFF_LEN = 0;                     // int32 [64] lengths
constexpr size_t ST_OFF_ERR = 256;                   // uint32 device error word
constexpr size_t ST_OFF_HIST = 512;                  // uint32 [64][4096] first-digit histograms
constexpr size_t ST_OFF_KEYS = ST_OFF_HIST + (size_t)ST_MAX_REQUESTS * IDX_BINS * 4;   // uint32 keys
constexpr size_t ST_BYTES = ST_OFF_KEYS + (size_t)ST_MAX_POSITIONS * 4;   // about 9 MiB
}  // namespace
}  // namespace hs

// Scratch of every call: one array per GPU that loads the library, held until
// the process exits.  Host code must not use this name as a device address; it
// uses the address cudaGetSymbolAddress returns (see the set-up below).
static __device__ __align__(256) unsigned char hs_static_scratch[hs::ST_BYTES];

namespace hs {
namespace {
constexpr int ST_MAX_DEVICES = 64;
unsigned char* g_scratch[ST_MAX_DEVICES] = {};   // device address of the array, per device
int g_num_sms[ST_MAX_DEVICES] = {};

struct TopkShared {
  int scan[2 * (RES_THREADS / 32 + 1)];
  int b1, above1, b2, above2;
};

__device__ __forceinline__ void digit_from_top(const uint32_t* h, int kneed, int* scan, int* out_b,
                                               int* out_above) {
  constexpr int PER = IDX_BINS / RES_THREADS;
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

// Exact top-k over the keys the score kernel left in the scratch array (the
// selection step of the decode path, without the cache update).  One CTA per
// request; output ascending, ties to the lower position, -1 past k_eff.  When
// the score kernel recorded an error (a bounded wait gave up, so some keys are
// missing), every entry becomes -1: no partial selection passes as a result.
__global__ void __launch_bounds__(RES_THREADS, 1)
    static_topk_kernel(const uint32_t* keys_all, const uint32_t* hist_all, const int32_t* lengths,
                       const unsigned int* err, long long stride, int top_k, int32_t* sel_out) {
  __shared__ uint32_t h[IDX_BINS];
  __shared__ TopkShared sh;
  const int tid = threadIdx.x;
  const int ri = blockIdx.x;
  const int K = top_k;
  const int N = lengths[ri];
  int32_t* sel = sel_out + (long long)ri * K;
  if (*reinterpret_cast<const volatile unsigned int*>(err) != 0u) {
    for (int i = tid; i < K; i += RES_THREADS) sel[i] = -1;
    return;
  }
  if (N <= K) {
    for (int i = tid; i < K; i += RES_THREADS) sel[i] = i < N ? i : -1;
    return;
  }
  const uint32_t* keys = keys_all + (long long)ri * stride;
  for (int b = tid; b < IDX_BINS; b += RES_THREADS) h[b] = hist_all[(long long)ri * IDX_BINS + b];
  __syncthreads();
  digit_from_top(h, K, sh.scan, &sh.b1, &sh.above1);
  const int b1 = sh.b1, above1 = sh.above1;
  for (int b = tid; b < IDX_BINS; b += RES_THREADS) h[b] = 0;
  __syncthreads();
  for (int i = tid; i < N; i += RES_THREADS) {
    const uint32_t v = keys[i];
    if ((int)(v >> 12) == b1) atomicAdd(&h[v & 4095u], 1u);
  }
  __syncthreads();
  digit_from_top(h, K - above1, sh.scan, &sh.b2, &sh.above2);
  const uint32_t vstar = ((uint32_t)b1 << 12) | (uint32_t)sh.b2;
  const int need_eq = K - (above1 + sh.above2);
  const int per = (N + RES_THREADS - 1) / RES_THREADS;
  const int j0 = min(N, tid * per), j1 = min(N, j0 + per);
  int n_gt = 0, n_eq = 0;
  for (int j = j0; j < j1; ++j) {
    const uint32_t v = keys[j];
    n_gt += v > vstar;
    n_eq += v == vstar;
  }
  const int2 before = block_exclusive_scan2<RES_THREADS>(n_gt, n_eq, sh.scan, nullptr, nullptr);
  int o = before.x + min(before.y, need_eq);
  int eq_rank = before.y;
  for (int j = j0; j < j1; ++j) {
    const uint32_t v = keys[j];
    bool take = v > vstar;
    if (v == vstar) {
      take = eq_rank < need_eq;
      ++eq_rank;
    }
    if (take && o < K) sel[o++] = j;
  }
}

struct Lengths {
  int32_t v[ST_MAX_REQUESTS];
};

// Puts the lengths (passed by value) where the score kernel reads them.
__global__ void static_lengths_kernel(Lengths len, int n_req, int32_t* dst) {
  if ((int)threadIdx.x < n_req) dst[threadIdx.x] = len.v[threadIdx.x];
}

}  // namespace

}  // namespace hs

extern "C" int hs_indexer_topk_static(int32_t n_req, int32_t n_max, int32_t d_idx, int32_t top_k,
                                      const int8_t* idx_keys, const int32_t* lengths, const int8_t* q_idx,
                                      int32_t* sel_out, int32_t device, void* stream) {
  using namespace hs;
  if (n_req < 0 || n_req > ST_MAX_REQUESTS)
    return set_static_error(HS_ERR_CAPACITY, "hs_indexer_topk_static: n_req above the maximum of 64");
  if (n_req == 0) return HS_OK;
  if (n_max < 1 || top_k < 1 || !idx_keys || !lengths || !q_idx || !sel_out)
    return set_static_error(HS_ERR_INVALID, "hs_indexer_topk_static: null buffer or empty size");
  if (d_idx != 16 && d_idx != 32 && d_idx != 64 && d_idx != 128 && d_idx != 256)
    return set_static_error(HS_ERR_INVALID, "hs_indexer_topk_static: d_idx must be 16, 32, 64, 128 or 256");
  if ((reinterpret_cast<uintptr_t>(idx_keys) & 15u) || (reinterpret_cast<uintptr_t>(q_idx) & 15u) ||
      (reinterpret_cast<uintptr_t>(sel_out) & 3u))
    return set_static_error(HS_ERR_INVALID, "hs_indexer_topk_static: misaligned buffer");
  const long long stride = ((long long)n_max + 3) & ~3LL;
  if ((long long)n_req * stride > ST_MAX_POSITIONS)
    return set_static_error(HS_ERR_CAPACITY,
                            "hs_indexer_topk_static: n_req * n_max (rounded up to 4) above the maximum of 2^21");
  Lengths len = {};
  for (int i = 0; i < n_req; ++i) {
    if (lengths[i] < 0 || lengths[i] > n_max)
      return set_static_error(HS_ERR_INVALID, "hs_indexer_topk_static: a length outside [0, n_max]");
    len.v[i] = lengths[i];
  }
  if (device < 0 || device >= ST_MAX_DEVICES)
    return set_static_error(HS_ERR_INVALID, "hs_indexer_topk_static: device out of range");

  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != device) {
    if (cudaSetDevice(device) != cudaSuccess) {
      (void)cudaGetLastError();
      return set_static_error(HS_ERR_CUDA, "hs_indexer_topk_static: cudaSetDevice failed");
    }
  }
  Geometry g = {};
  g.n_layers = 1;
  g.max_requests = n_req;
  g.max_context = n_max;
  g.d_idx = d_idx;
  g.top_k = top_k;
  const size_t smem = score_smem_bytes(g);
  // One-time set-up per device (the device is current): the array's device
  // address, the SM count and the score kernel's shared-memory allowance.
  if (g_scratch[device] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, hs_static_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return set_static_error(HS_ERR_CUDA, "hs_indexer_topk_static: cudaGetSymbolAddress failed");
    }
    if (cudaDeviceGetAttribute(&g_num_sms[device], cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      (void)cudaGetLastError();
      return set_static_error(HS_ERR_CUDA, "hs_indexer_topk_static: device query failed");
    }
    g_scratch[device] = static_cast<unsigned char*>(ptr);
  }
  // the score kernel's shared memory depends on n_req (its per-request table)
  if (prepare_score(g, smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return set_static_error(HS_ERR_CUDA, "hs_indexer_topk_static: kernel set-up failed");
  }
  unsigned char* scratch = g_scratch[device];
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* dlen = reinterpret_cast<int32_t*>(scratch + ST_OFF_LEN);
  uint32_t* dhist = reinterpret_cast<uint32_t*>(scratch + ST_OFF_HIST);
  uint32_t* dkeys = reinterpret_cast<uint32_t*>(scratch + ST_OFF_KEYS);
  unsigned int* derr = reinterpret_cast<unsigned int*>(scratch + ST_OFF_ERR);
  // what must start at zero: the histograms (the array keeps the previous call's contents)
  static_lengths_kernel<<<1, ST_MAX_REQUESTS, 0, st>>>(len, n_req, dlen);
  if (cudaGetLastError() != cudaSuccess || cudaMemsetAsync(dhist, 0, (size_t)n_req * IDX_BINS * 4, st) != cudaSuccess ||
      cudaMemsetAsync(derr, 0, 4, st) != cudaSuccess) {
    (void)cudaGetLastError();
    return set_static_error(HS_ERR_CUDA, "hs_indexer_topk_static: enqueue failed");
  }
  DecodeParams p = {};
  p.g = g;
  p.s.idx_keys = const_cast<int8_t*>(idx_keys);
  p.s.length = dlen;
  p.s.scores = dkeys;
  p.s.hist = dhist;
  p.s.dev_error = derr;
  p.layer = 0;
  p.n_req = n_req;
  p.req_ids = nullptr;
  p.q_idx = q_idx;
  p.score_stride = stride;
  p.score_grid = g_num_sms[device];
  if (launch_score(p, smem, st) != cudaSuccess) {
    (void)cudaGetLastError();
    return set_static_error(HS_ERR_CUDA, "hs_indexer_topk_static: score launch failed");
  }
  static_topk_kernel<<<n_req, RES_THREADS, 0, st>>>(dkeys, dhist, dlen, derr, stride, top_k, sel_out);
  if (cudaGetLastError() != cudaSuccess)
    return set_static_error(HS_ERR_CUDA, "hs_indexer_topk_static: top-k launch failed");
  return HS_OK;
}

extern "C" int hs_indexer_topk_static_error(int32_t device, uint32_t* out) {
  using namespace hs;
  if (!out) return set_static_error(HS_ERR_INVALID, "hs_indexer_topk_static_error: null argument");
  *out = 0;
  if (device < 0 || device >= ST_MAX_DEVICES)
    return set_static_error(HS_ERR_INVALID, "hs_indexer_topk_static_error: device out of range");
  if (g_scratch[device] == nullptr) return HS_OK;   // no call has run on this device
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != device) {
    if (cudaSetDevice(device) != cudaSuccess) {
      (void)cudaGetLastError();
      return set_static_error(HS_ERR_CUDA, "hs_indexer_topk_static_error: cudaSetDevice failed");
    }
  }
  unsigned int word = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(&word, hs_static_scratch, sizeof(word), ST_OFF_ERR, cudaMemcpyDeviceToHost) !=
          cudaSuccess) {
    (void)cudaGetLastError();
    return set_static_error(HS_ERR_CUDA, "hs_indexer_topk_static_error: reading the error word failed");
  }
  *out = word;
  if (word) return set_static_error(HS_ERR_DEVICE, "hs_indexer_topk_static: the last call's kernels set an error");
  return HS_OK;
}
