// Host side of the C ABI declared in include/hs.h: configuration checks,
// allocation of the two memory tiers and the cache metadata, argument checks
// and kernel launches, counters, snapshots and optional per-kernel timing.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <sys/mman.h>
#include <unistd.h>
#include <new>
#include <string>

#include "hs_internal.cuh"

namespace {

thread_local std::string g_create_error;

int set_err(hs_handle* h, int code, const std::string& msg) {
  if (h) h->last_error = msg;
  else g_create_error = msg;
  return code;
}

int cuda_fail(hs_handle* h, cudaError_t e, const char* what) {
  std::string msg = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  (void)cudaGetLastError();
  return set_err(h, HS_ERR_CUDA, msg);
}

bool is_pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

#ifndef MADV_COLLAPSE
#define MADV_COLLAPSE 25   // Linux 6.1+: synchronous collapse of a range into transparent huge pages
#endif

// Bytes backed by transparent huge pages in the anonymous mappings that overlap
// [a, a + n), from /proc/self/smaps (0 where it cannot be read).
size_t huge_bytes_in(const void* a, size_t n) {
  FILE* f = std::fopen("/proc/self/smaps", "r");
  if (!f) return 0;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(a), hi = lo + n;
  char line[512];
  bool in = false;
  unsigned long long kb = 0;
  while (std::fgets(line, sizeof line, f)) {
    unsigned long s0 = 0, s1 = 0;
    const char* dash = std::strchr(line, '-');
    const char* space = std::strchr(line, ' ');
    if (dash && space && dash < space && std::sscanf(line, "%lx-%lx", &s0, &s1) == 2) {
      in = s0 < hi && s1 > lo;   // a mapping's header line
    } else if (in && std::strncmp(line, "AnonHugePages:", 14) == 0) {
      kb += std::strtoull(line + 14, nullptr, 10);
    }
  }
  std::fclose(f);
  return (size_t)std::min<unsigned long long>(kb * 1024ull, n);
}

// Returns "" when the configuration is one the kernels support, else the reason.
std::string check_config(const hs_config_t& c) {
  if (c.n_layers < 1) return "n_layers must be >= 1";
  if (c.max_requests < 1 || c.max_requests > 4096) return "max_requests must be in [1, 4096]";
  if (c.max_context < 1 || c.max_context > HS_MAX_CONTEXT) return "max_context must be in [1, HS_MAX_CONTEXT]";
  if (!is_pow2_in(c.d_idx, 16, 256)) return "d_idx must be one of 16, 32, 64, 128, 256";
  if (c.top_k < 1 || c.top_k > 8192) return "top_k must be in [1, 8192]";
  if (c.hot_slots < c.top_k || c.hot_slots > 16384) return "hot_slots must be in [top_k, 16384]";
  if (c.hot_slots % 4 != 0) return "hot_slots must be a multiple of 4";
  if (!(c.softmax_scale >= 0.f) || !std::isfinite(c.softmax_scale)) return "softmax_scale must be finite and >= 0";
  if (c.fetch_mode < 0 || c.fetch_mode > 2) return "fetch_mode must be 0, 1 or 2";
  if (c.replacement != HS_REPLACE_LRU && c.replacement != HS_REPLACE_FIFO && c.replacement != HS_REPLACE_RANDOM)
    return "replacement must be HS_REPLACE_LRU (0), HS_REPLACE_FIFO (1) or HS_REPLACE_RANDOM (2)";
  if (c.write_allocate != 0 && c.write_allocate != 1) return "write_allocate must be 0 or 1";
  if (c.index_share < 0 || c.index_share > c.n_layers) return "index_share must be in [0, n_layers]";
  if (c.share_prefetch != 0 && c.share_prefetch != 1) return "share_prefetch must be 0 or 1";
  if (c.index_share > 1 && c.shared_kv) return "index_share > 1 is supported for GQA rows";
  if (c.idx_heads < 0 || c.idx_heads > 8 || (c.idx_heads > 1 && (c.idx_heads & (c.idx_heads - 1))))
    return "idx_heads must be 0, 1, 2, 4 or 8";
  if (c.idx_heads > 1 && c.d_idx != 64 && c.d_idx != 128)
    return "the multi-head indexer (idx_heads > 1) needs d_idx 64 or 128";
  if (c.write_allocate && c.top_k >= c.hot_slots)
    return "write_allocate needs top_k < hot_slots (the appended token needs a slot of its own)";
  if (c.page_size < 0 || c.page_size > 64 || (c.page_size > 1 && (c.page_size & (c.page_size - 1))))
    return "page_size must be 0, 1, 2, 4, 8, 16, 32 or 64";
  if (c.page_size > 1) {
    if (c.shared_kv) return "page_size > 1 is supported for GQA rows";
    if (c.d_idx != 64 && c.d_idx != 128) return "page_size > 1 needs d_idx 64 or 128";
    if (c.idx_heads > 1 || c.index_share > 1 || c.write_allocate)
      return "page_size > 1 excludes idx_heads > 1, index_share > 1 and write_allocate";
    if (c.top_k % c.page_size != 0) return "page_size > 1 needs top_k % page_size == 0";
    if (c.hot_slots % (4 * c.page_size) != 0) return "page_size > 1 needs hot_slots % (4 * page_size) == 0";
  }
  if (c.shared_kv == 0) {
    if (c.d_qk != 128 || c.d_v != 128) return "GQA rows: d_qk = d_v = 128 required";
    if (!is_pow2_in(c.h_kv, 1, 8)) return "GQA rows: h_kv must be one of 1, 2, 4, 8";
    if (c.h_q < c.h_kv || c.h_q % c.h_kv != 0) return "GQA rows: h_q must be a multiple of h_kv";
    if (!is_pow2_in(c.h_q / c.h_kv, 1, 16)) return "GQA rows: h_q / h_kv must be one of 1, 2, 4, 8, 16";
  } else if (c.shared_kv == 1) {
    if (c.h_kv != 1 || c.d_qk != 576 || c.d_v != 512)
      return "latent rows: h_kv = 1, d_qk = 576 (the row, read as K), d_v = 512 (its first 512 dims, read as V)";
    if (c.h_q != 16 && c.h_q != 32 && c.h_q != 64 && c.h_q != 128) return "latent rows: h_q must be 16, 32, 64 or 128";
  } else {
    return "shared_kv must be 0 or 1";
  }
  return "";
}

void free_all(hs_handle* h) {
  for (void* p : h->dev_allocs) cudaFree(p);
  h->dev_allocs.clear();
  if (h->host_kv_host) {
    if (h->host_map_base) {
      cudaHostUnregister(h->host_kv_host);
      munmap(h->host_map_base, h->host_map_bytes);
    } else {
      cudaFreeHost(h->host_kv_host);
    }
  }
  h->host_kv_host = nullptr;
  h->host_map_base = nullptr;
  for (auto& t : h->timed) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  h->timed.clear();
  for (cudaEvent_t e : h->event_pool) cudaEventDestroy(e);
  h->event_pool.clear();
}

struct FaultInject {
  bool host = false, dev = false, noready = false;
  FaultInject() {
    const char* v = std::getenv("HS_FAULT_INJECT");
    if (v) {
      host = std::strcmp(v, "hostalloc") == 0;
      dev = std::strcmp(v, "devalloc") == 0;
      noready = std::strcmp(v, "noready") == 0;
    }
  }
};

template <typename T>
cudaError_t dev_alloc(hs_handle* h, T** p, size_t bytes, FaultInject& fi) {
  if (fi.dev) {
    fi.dev = false;
    return cudaErrorMemoryAllocation;
  }
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
  if (e == cudaSuccess) {
    h->dev_allocs.push_back(q);
    *p = static_cast<T*>(q);
  }
  return e;
}

cudaEvent_t take_event(hs_handle* h) {
  if (!h->event_pool.empty()) {
    cudaEvent_t e = h->event_pool.back();
    h->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one launch with events when timing is on.
template <typename F>
cudaError_t timed_launch(hs_handle* h, int kind, cudaStream_t st, F&& launch) {
  if (!h->timing) return launch();
  cudaEvent_t a = take_event(h), b = take_event(h);
  if (!a || !b) return launch();
  // Under stream capture the events become external event-record nodes, so
  // they can still be timed after the graph is replayed.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  const unsigned flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  cudaEventRecordWithFlags(a, st, flags);
  cudaError_t e = launch();
  cudaEventRecordWithFlags(b, st, flags);
  h->timed.push_back({kind, a, b});
  return e;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Makes the handle's device current without a call when it already is (keeps
// the enqueue path free of anything but launches, e.g. under stream capture).
void use_device(const hs_handle* h) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != h->cfg.device) cudaSetDevice(h->cfg.device);
}

}  // namespace

int hs::set_static_error(int code, const char* msg) {
  g_create_error = msg;
  return code;
}

extern "C" {

const char* hs_status_string(int32_t s) {
  switch (s) {
    case HS_OK: return "HS_OK";
    case HS_ERR_INVALID: return "HS_ERR_INVALID";
    case HS_ERR_CONFIG: return "HS_ERR_CONFIG";
    case HS_ERR_OOM: return "HS_ERR_OOM";
    case HS_ERR_CAPACITY: return "HS_ERR_CAPACITY";
    case HS_ERR_CUDA: return "HS_ERR_CUDA";
    case HS_ERR_DEVICE: return "HS_ERR_DEVICE";
    default: return "HS_ERR_UNKNOWN";
  }
}

const char* hs_last_error(const hs_handle_t* h) { return h ? h->last_error.c_str() : g_create_error.c_str(); }

int32_t hs_row_elems(const hs_config_t* c) {
  if (!c || !check_config(*c).empty()) return 0;
  return c->shared_kv ? c->d_qk : c->h_kv * (c->d_qk + c->d_v);
}

int hs_create(const hs_config_t* cfg, hs_handle_t** out) {
  g_create_error.clear();
  if (!cfg || !out) return set_err(nullptr, HS_ERR_INVALID, "hs_create: null argument");
  *out = nullptr;
  const std::string why = check_config(*cfg);
  if (!why.empty()) return set_err(nullptr, HS_ERR_CONFIG, "hs_create: " + why);

  hs_handle* h = new (std::nothrow) hs_handle();
  if (!h) return set_err(nullptr, HS_ERR_OOM, "hs_create: out of host memory");
  h->cfg = *cfg;
  hs::Geometry& g = h->g;
  g.n_layers = cfg->n_layers;
  g.max_requests = cfg->max_requests;
  g.max_context = cfg->max_context;
  g.h_q = cfg->h_q;
  g.h_kv = cfg->h_kv;
  g.d_qk = cfg->d_qk;
  g.d_v = cfg->d_v;
  g.shared_kv = cfg->shared_kv;
  g.d_idx = cfg->d_idx;
  g.top_k = cfg->top_k;
  g.hot_slots = cfg->hot_slots;
  g.row_elems = hs_row_elems(cfg);
  g.row_bytes = 2 * g.row_elems;
  g.v_off = cfg->shared_kv ? 0 : cfg->h_kv * cfg->d_qk;
  g.idx_heads = cfg->idx_heads > 1 ? cfg->idx_heads : 1;
  g.page_size = cfg->page_size > 1 ? cfg->page_size : 1;
  g.page_shift = 0;
  while ((1 << g.page_shift) < g.page_size) ++g.page_shift;
  g.max_pages = (cfg->max_context + g.page_size - 1) / g.page_size;
  const float scale = cfg->softmax_scale > 0.f ? cfg->softmax_scale : 1.0f / std::sqrt((float)cfg->d_qk);
  h->scale_log2 = scale * 1.4426950408889634f;

  auto fail_free = [&](int code, const std::string& msg) {
    free_all(h);
    delete h;
    return set_err(nullptr, code, msg);
  };

  cudaError_t e = cudaSetDevice(cfg->device);
  if (e != cudaSuccess) {
    std::string msg = std::string("hs_create: cudaSetDevice: ") + cudaGetErrorName(e);
    (void)cudaGetLastError();
    delete h;
    return set_err(nullptr, HS_ERR_CUDA, msg);
  }
  int smem_optin = 0, cluster_ok = 0;
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, cfg->device);
  cudaDeviceGetAttribute(&cluster_ok, cudaDevAttrClusterLaunch, cfg->device);
  if (!cluster_ok) return fail_free(HS_ERR_CONFIG, "hs_create: device has no thread-block cluster launch");

  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, cfg->device);
  h->score_stride = ((long long)cfg->max_context + 3) & ~3LL;
  h->sel_smem = hs::select_smem_bytes(g);
  h->att_smem = hs::attention_smem_bytes(g);
  h->att_parts = hs::attention_parts(g);
  if (h->num_sms < 2)
    return fail_free(HS_ERR_CONFIG, "hs_create: the select kernel needs at least two SMs");
  if (h->sel_smem > (size_t)smem_optin)
    return fail_free(HS_ERR_CONFIG,
                     "hs_create: top_k / hot_slots / max_requests too large for the select kernel's shared memory");
  if (h->att_smem > (size_t)smem_optin)
    return fail_free(HS_ERR_CONFIG,
                     "hs_create: rows or max_requests too large for the attention kernel's shared memory");

  const size_t R = cfg->max_requests, Lr = cfg->n_layers, N = cfg->max_context, B = cfg->hot_slots;
  const size_t K = cfg->top_k;
  h->host_bytes = R * Lr * N * (size_t)g.row_bytes;
  h->hot_bytes = R * Lr * B * (size_t)g.row_bytes;
  h->index_bytes = R * Lr * N * (size_t)g.d_idx;
  const size_t pbound_bytes = g.page_size > 1 ? R * Lr * (size_t)g.max_pages * 2 * g.d_idx : 16;
  if (g.page_size > 1) h->index_bytes += pbound_bytes;

  FaultInject fi;
  h->fault = fi.noready ? 1 : 0;
  // D1: authoritative copy in pinned, mapped host memory
  if (fi.host) return fail_free(HS_ERR_OOM, "hs_create: pinned host allocation failed (injected)");
  // Anonymous memory in whole transparent huge pages, then pinned and mapped:
  // the missed rows are read at random positions, and a read of a row on a huge
  // page takes about half as long as one on base pages (a latency the attention
  // kernel waits for).  The store is faulted in first; whatever the kernel backed
  // with base pages is then collapsed synchronously (MADV_COLLAPSE, which
  // compacts memory as needed); the coverage is reported by hs_stats.  Falls
  // back to cudaHostAlloc where mapping or registration fails.
  void* hp = nullptr;
  {
    const size_t align = (size_t)512 << 20;   // the largest huge page (64 KB base pages); a multiple of the rest
    const size_t span = (h->host_bytes + align - 1) / align * align;
    const size_t len = span + align;
    void* raw = mmap(nullptr, len, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (raw != MAP_FAILED) {
      void* a = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(raw) + align - 1) & ~(uintptr_t)(align - 1));
      (void)madvise(a, span, MADV_HUGEPAGE);
      const long pg = sysconf(_SC_PAGESIZE);
      const size_t step = pg > 0 ? (size_t)pg : 4096;
      for (size_t off = 0; off < span; off += step) static_cast<volatile unsigned char*>(a)[off] = 0;
      if (huge_bytes_in(a, span) < span) (void)madvise(a, span, MADV_COLLAPSE);
      h->host_huge_bytes = std::min(huge_bytes_in(a, span), h->host_bytes);
      if (cudaHostRegister(a, h->host_bytes, cudaHostRegisterMapped | cudaHostRegisterPortable) == cudaSuccess) {
        hp = a;
        h->host_map_base = raw;
        h->host_map_bytes = len;
      } else {
        (void)cudaGetLastError();
        munmap(raw, len);
      }
    }
  }
  e = hp ? cudaSuccess : cudaHostAlloc(&hp, h->host_bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail_free(HS_ERR_OOM, std::string("hs_create: cudaHostAlloc of ") + std::to_string(h->host_bytes) +
                                     " bytes failed: " + cudaGetErrorName(e));
  }
  h->host_kv_host = static_cast<uint16_t*>(hp);
  void* dp = nullptr;
  e = cudaHostGetDevicePointer(&dp, hp, 0);
  if (e != cudaSuccess) return fail_free(HS_ERR_CUDA, "hs_create: cudaHostGetDevicePointer failed");
  h->s.host_kv = static_cast<uint16_t*>(dp);

  hs::DeviceState& s = h->s;
  size_t meta = 0;
  struct A {
    void** p;
    size_t bytes;
    bool meta;
  };
  const A allocs[] = {
      {(void**)&s.hot, h->hot_bytes, false},
      {(void**)&s.idx_keys, R * Lr * N * (size_t)g.d_idx, false},
      {(void**)&s.pbound, pbound_bytes, false},
      {(void**)&s.page, R * Lr * N * 4, true},
      {(void**)&s.reverse, R * Lr * B * 4, true},
      {(void**)&s.stamp, R * Lr * B * 4, true},
      {(void**)&s.order, R * Lr * B * 4, true},
      {(void**)&s.length, R * Lr * 4, true},
      {(void**)&s.step, R * Lr * 4, true},
      {(void**)&s.hits, R * Lr * 8, true},
      {(void**)&s.misses, R * Lr * 8, true},
      {(void**)&s.glob, 8 * 8, true},
      {(void**)&s.att_cta, (size_t)h->num_sms * 16, false},
      {(void**)&s.dev_error, 16, true},
      {(void**)&s.scores, R * (size_t)h->score_stride * 4, false},
      {(void**)&s.hist, R * (size_t)hs::IDX_BINS * 4, false},
      {(void**)&s.cand_thr, R * Lr * 4, true},
      {(void**)&s.cand_cnt, R * 4, false},
      {(void**)&s.cand, R * 2 * K * 8, false},
      {(void**)&s.cand_slot, R * 2 * K * 4, false},
      {(void**)&s.sel, R * K * 4, false},
      {(void**)&s.slot_of_sel, R * K * 4, false},
      {(void**)&s.part_o, R * (size_t)h->att_parts * g.h_q * g.d_v * 4, false},
      {(void**)&s.part_ml, R * (size_t)h->att_parts * g.h_q * 2 * 4, false},
      {(void**)&s.att_nparts, R * 8 * 4, false},
      {(void**)&s.call_n, R * 4, false},
      {(void**)&s.app_counter, R * 4, false},
      {(void**)&s.tiles_done, R * 4, false},
      {(void**)&s.ready, R * 4, false},
      {(void**)&s.miss_cnt, R * 4, false},
      {(void**)&s.att_done, R * 4, false},
      {(void**)&s.miss_pos, R * K * 4, false},
      {(void**)&s.sync, 32, false},
      {(void**)&s.sh_sel, cfg->index_share > 1 ? R * Lr * K * 4 : 16, false},
      {(void**)&s.sh_slots, cfg->index_share > 1 ? R * Lr * K * 4 : 16, false},
      {(void**)&s.sh_kk, R * Lr * 4, false},
      {(void**)&s.sh_pend, R * Lr * 4, false},
      {(void**)&s.sh_armed, R * Lr * 4, false},
#ifdef HS_WITH_TRACE
      {(void**)&h->trace, 2 * (size_t)hs::TRACE_KERNELS * hs::TRACE_CTAS * hs::TRACE_POINTS * 8, false},
#endif
  };
  for (const A& a : allocs) {
    e = dev_alloc(h, a.p, a.bytes, fi);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return fail_free(HS_ERR_OOM, std::string("hs_create: device allocation of ") + std::to_string(a.bytes) +
                                       " bytes failed: " + cudaGetErrorName(e));
    }
    if (a.meta) meta += a.bytes;
    // every allocation starts zeroed (the specific initial values follow)
    if (cudaMemsetAsync(*a.p, 0, a.bytes, 0) != cudaSuccess) {
      (void)cudaGetLastError();
      return fail_free(HS_ERR_CUDA, "hs_create: clearing a device allocation failed");
    }
  }
  h->meta_bytes = meta;

  // initial state: empty cache everywhere
  bool ok = cudaMemset(s.page, 0xff, R * Lr * N * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.reverse, 0xff, R * Lr * B * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.stamp, 0xff, R * Lr * B * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.length, 0, R * Lr * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.step, 0, R * Lr * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.hits, 0, R * Lr * 8) == cudaSuccess;
  ok = ok && cudaMemset(s.misses, 0, R * Lr * 8) == cudaSuccess;
  ok = ok && cudaMemset(s.glob, 0, 64) == cudaSuccess;
  ok = ok && cudaMemset(s.dev_error, 0, 16) == cudaSuccess;
  ok = ok && cudaMemset(s.slot_of_sel, 0, R * K * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.att_nparts, 0, R * 8 * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.call_n, 0, R * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.hist, 0, R * (size_t)hs::IDX_BINS * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.cand_thr, 0, R * Lr * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.cand_cnt, 0, R * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.app_counter, 0, R * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.tiles_done, 0, R * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.ready, 0, R * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.sync, 0, 32) == cudaSuccess;
  ok = ok && cudaMemset(s.sh_armed, 0, R * Lr * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.sh_kk, 0, R * Lr * 4) == cudaSuccess;
  ok = ok && cudaMemset(s.sh_pend, 0xff, R * Lr * 4) == cudaSuccess;
#ifdef HS_WITH_TRACE
  ok = ok && cudaMemset(h->trace, 0, 2 * (size_t)hs::TRACE_KERNELS * hs::TRACE_CTAS * hs::TRACE_POINTS * 8) ==
                 cudaSuccess;
#endif
  ok = ok && hs::launch_init_order(s.order, (long long)(R * Lr), (int)B, 0) == cudaSuccess;
  if (!ok) return fail_free(HS_ERR_CUDA, "hs_create: initialising the metadata failed");
  if ((e = hs::prepare_select(g, h->sel_smem)) != cudaSuccess ||
      (e = hs::prepare_attention(g, h->att_smem)) != cudaSuccess)
    return fail_free(HS_ERR_CUDA, std::string("hs_create: kernel set-up failed: ") + cudaGetErrorName(e));
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_free(HS_ERR_CUDA, std::string("hs_create: ") + cudaGetErrorName(e));
  *out = h;
  return HS_OK;
}

void hs_destroy(hs_handle_t* h) {
  if (!h) return;
  cudaSetDevice(h->cfg.device);
  cudaDeviceSynchronize();
#ifdef HS_WITH_TRACE
  if (const char* path = std::getenv("HS_TRACE_OUT")) {
    std::vector<unsigned long long> t(2 * (size_t)hs::TRACE_KERNELS * hs::TRACE_CTAS * hs::TRACE_POINTS);
    if (cudaMemcpy(t.data(), h->trace, t.size() * 8, cudaMemcpyDeviceToHost) == cudaSuccess)
      if (FILE* f = std::fopen(path, "wb")) {
        std::fwrite(t.data(), 8, t.size(), f);
        std::fclose(f);
      }
  }
#endif
  free_all(h);
  delete h;
}

int hs_append(hs_handle_t* h, int32_t layer, int32_t n_req, const int32_t* req_ids, int32_t n_tok,
              const void* kv_rows, const int8_t* idx_keys, void* stream) {
  if (!h) return HS_ERR_INVALID;
  if (layer < 0 || layer >= h->cfg.n_layers) return set_err(h, HS_ERR_INVALID, "hs_append: layer out of range");
  if (n_req < 0 || n_req > h->cfg.max_requests) return set_err(h, HS_ERR_INVALID, "hs_append: n_req out of range");
  if (n_tok < 0) return set_err(h, HS_ERR_INVALID, "hs_append: n_tok < 0");
  if (n_tok > h->cfg.max_context)
    return set_err(h, HS_ERR_CAPACITY, "hs_append: n_tok exceeds max_context");
  if (n_req == 0 || n_tok == 0) return HS_OK;
  if (!kv_rows || !idx_keys) return set_err(h, HS_ERR_INVALID, "hs_append: null buffer");
  if (!aligned16(kv_rows) || !aligned16(idx_keys))
    return set_err(h, HS_ERR_INVALID, "hs_append: kv_rows and idx_keys must be 16-byte aligned");
  use_device(h);
  hs::AppendParams p;
  p.g = h->g;
  p.s = h->s;
  p.layer = layer;
  p.n_req = n_req;
  p.n_tok = n_tok;
  p.req_ids = req_ids;
  p.kv_rows = static_cast<const uint16_t*>(kv_rows);
  p.keys = idx_keys;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = timed_launch(h, HS_K_APPEND, st, [&] {
    cudaError_t r = hs::launch_append(p, st);
    if (r == cudaSuccess && p.g.page_shift > 0) r = hs::launch_page_bounds(p, st);   // bounds of the touched pages
    return r;
  });
  if (e != cudaSuccess) return cuda_fail(h, e, "hs_append: launch");
  ++h->append_calls;
  return HS_OK;
}

int hs_decode_layer(hs_handle_t* h, int32_t layer, int32_t n_req, const int32_t* req_ids, const int8_t* q_idx,
                    const void* q, void* out, int32_t* sel_out, const void* new_kv_rows,
                    const int8_t* new_idx_keys, void* stream) {
  if (!h) return HS_ERR_INVALID;
  if (layer < 0 || layer >= h->cfg.n_layers)
    return set_err(h, HS_ERR_INVALID, "hs_decode_layer: layer out of range");
  if (n_req < 0 || n_req > h->cfg.max_requests)
    return set_err(h, HS_ERR_INVALID, "hs_decode_layer: n_req out of range");
  if (n_req == 0) return HS_OK;
  if (!q_idx || !q || !out) return set_err(h, HS_ERR_INVALID, "hs_decode_layer: null buffer");
  if (!aligned16(q_idx)) return set_err(h, HS_ERR_INVALID, "hs_decode_layer: q_idx must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(q) & 1u) || (reinterpret_cast<uintptr_t>(out) & 1u) ||
      (reinterpret_cast<uintptr_t>(sel_out) & 3u))
    return set_err(h, HS_ERR_INVALID, "hs_decode_layer: misaligned q / out / sel_out");
  if ((new_kv_rows == nullptr) != (new_idx_keys == nullptr))
    return set_err(h, HS_ERR_INVALID, "hs_decode_layer: new_kv_rows and new_idx_keys go together");
  if (new_kv_rows && (!aligned16(new_kv_rows) || !aligned16(new_idx_keys)))
    return set_err(h, HS_ERR_INVALID, "hs_decode_layer: new_kv_rows and new_idx_keys must be 16-byte aligned");
  const int G = h->cfg.index_share > 1 ? h->cfg.index_share : 1;
  if (G > 1 && !new_kv_rows)
    return set_err(h, HS_ERR_INVALID, "hs_decode_layer: with index_share > 1 every call appends its token "
                                      "(new_kv_rows, new_idx_keys)");
  use_device(h);
  hs::DecodeParams p;
  p.g = h->g;
  p.s = h->s;
  p.layer = layer;
  p.n_req = n_req;
  p.req_ids = req_ids;
  p.q_idx = q_idx;
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  p.sel_out = sel_out;
  p.new_kv = static_cast<const uint16_t*>(new_kv_rows);
  p.new_keys = new_idx_keys;
  p.scale_log2 = h->scale_log2;
  p.score_stride = h->score_stride;
  p.score_grid = h->num_sms;
  p.att_parts = h->att_parts;
  p.att_grid = h->num_sms;
  // latent rows are read by every head group's CTAs: RESOLVE pulls them (once)
  p.fetch_mode = h->cfg.shared_kv ? 1 : (h->cfg.fetch_mode == 1 ? 1 : 0);
  p.replacement = h->cfg.replacement;
  p.replacement_seed = h->cfg.replacement_seed;
  p.sel_grid = h->num_sms;
  p.n_resolvers = std::min(std::min(n_req, hs::SEL_MAX_RESOLVERS), h->num_sms - 1);
  p.publish = h->cfg.shared_kv ? 0 : 1;   // the chunked GQA kernel starts on published requests
  p.fault = h->fault;
  p.write_allocate = h->cfg.write_allocate;
  const bool lead = layer % G == 0;
  p.role = lead ? hs::ROLE_SELECT : hs::ROLE_GIVEN;
  p.n_follow = lead ? std::min(G, h->cfg.n_layers - layer) - 1 : 0;
  p.share_prefetch = h->cfg.share_prefetch;
#ifdef HS_WITH_TRACE
  p.trace = h->trace;
#endif
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // a follower of a prefetching group only appends its token and attends
  const bool follow = !lead && p.share_prefetch;
  cudaError_t e = timed_launch(h, HS_K_SELECT, st, [&] {
    return follow ? hs::launch_follow(p, st) : hs::launch_select(p, h->sel_smem, st);
  });
  if (e != cudaSuccess) return cuda_fail(h, e, "hs_decode_layer: select launch");
  e = timed_launch(h, HS_K_ATTENTION, st, [&] { return hs::launch_attention(p, h->att_smem, st); });
  if (e != cudaSuccess) return cuda_fail(h, e, "hs_decode_layer: attention launch");
  ++h->decode_calls;
  if (new_kv_rows) ++h->append_calls;
  return HS_OK;
}

int hs_stats(hs_handle_t* h, hs_stats_t* out) {
  if (!h || !out) return HS_ERR_INVALID;
  cudaSetDevice(h->cfg.device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e, "hs_stats: synchronize");
  const size_t RL = (size_t)h->cfg.max_requests * h->cfg.n_layers;
  std::vector<unsigned long long> hits(RL), misses(RL), glob(8), cta(2 * (size_t)h->num_sms);
  unsigned int err = 0;
  if ((e = cudaMemcpy(hits.data(), h->s.hits, RL * 8, cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemcpy(misses.data(), h->s.misses, RL * 8, cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemcpy(glob.data(), h->s.glob, 64, cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemcpy(cta.data(), h->s.att_cta, cta.size() * 8, cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemcpy(&err, h->s.dev_error, 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(h, e, "hs_stats: copy");
  std::memset(out, 0, sizeof(*out));
  for (size_t i = 0; i < RL; ++i) {
    out->hits += hits[i];
    out->misses += misses[i];
  }
  out->h2d_bytes = glob[0];
  out->d2h_bytes = glob[1];
  out->decode_calls = h->decode_calls;
  out->append_calls = h->append_calls;
  out->host_bytes = h->host_bytes;
  out->hot_bytes = h->hot_bytes;
  out->index_bytes = h->index_bytes;
  out->meta_bytes = h->meta_bytes;
  out->full_selects = glob[2];
  out->att_host_wait_ns = glob[4];
  out->att_host_stages = glob[5];
  out->att_hbm_wait_ns = glob[6];
  out->att_hbm_stages = glob[7];
  // the latest launch's CTA timeline (a CTA that has not run yet holds zeros)
  {
    std::vector<unsigned long long> ends;
    unsigned long long first = ~0ull, last = 0;
    for (int b = 0; b < h->num_sms; ++b) {
      const unsigned long long t0 = cta[2 * b], t1 = cta[2 * b + 1];
      if (t0 == 0 || t1 < t0) continue;
      first = std::min(first, t0);
      last = std::max(last, t1);
      ends.push_back(t1);
    }
    if (!ends.empty()) {
      std::sort(ends.begin(), ends.end());
      out->att_last_span_ns = last - first;
      out->att_last_median_ns = ends[ends.size() / 2] - first;
    }
  }
  out->host_huge_bytes = h->host_huge_bytes;
  out->device_error = err;
  if (err) return set_err(h, HS_ERR_DEVICE, "hs_stats: device error word " + std::to_string(err));
  return HS_OK;
}

int hs_snapshot(hs_handle_t* h, int32_t req, int32_t layer, int32_t* page, int32_t n_page, int32_t* reverse,
                int32_t* stamp, int32_t* order, int64_t* scalars) {
  if (!h) return HS_ERR_INVALID;
  if (req < 0 || req >= h->cfg.max_requests || layer < 0 || layer >= h->cfg.n_layers)
    return set_err(h, HS_ERR_INVALID, "hs_snapshot: request or layer out of range");
  if (page && (n_page < 0 || n_page > h->cfg.max_context))
    return set_err(h, HS_ERR_INVALID, "hs_snapshot: n_page out of range");
  cudaSetDevice(h->cfg.device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e, "hs_snapshot: synchronize");
  const size_t rl = (size_t)req * h->cfg.n_layers + layer;
  const size_t B = h->cfg.hot_slots;
  if (page && n_page > 0 &&
      (e = cudaMemcpy(page, h->s.page + rl * h->cfg.max_context, (size_t)n_page * 4, cudaMemcpyDeviceToHost)) !=
          cudaSuccess)
    return cuda_fail(h, e, "hs_snapshot: page");
  if (reverse && (e = cudaMemcpy(reverse, h->s.reverse + rl * B, B * 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(h, e, "hs_snapshot: reverse");
  if (stamp && (e = cudaMemcpy(stamp, h->s.stamp + rl * B, B * 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(h, e, "hs_snapshot: stamp");
  if (order && (e = cudaMemcpy(order, h->s.order + rl * B, B * 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(h, e, "hs_snapshot: order");
  if (scalars) {
    int32_t len = 0, step = 0;
    unsigned long long hi = 0, mi = 0;
    if ((e = cudaMemcpy(&len, h->s.length + rl, 4, cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemcpy(&step, h->s.step + rl, 4, cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemcpy(&hi, h->s.hits + rl, 8, cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemcpy(&mi, h->s.misses + rl, 8, cudaMemcpyDeviceToHost)) != cudaSuccess)
      return cuda_fail(h, e, "hs_snapshot: scalars");
    scalars[0] = len;
    scalars[1] = step;
    scalars[2] = (int64_t)hi;
    scalars[3] = (int64_t)mi;
  }
  return HS_OK;
}

int hs_reset_request(hs_handle_t* h, int32_t req, void* stream) {
  if (!h) return HS_ERR_INVALID;
  if (req < 0 || req >= h->cfg.max_requests)
    return set_err(h, HS_ERR_INVALID, "hs_reset_request: request out of range");
  use_device(h);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t L = h->cfg.n_layers, N = h->cfg.max_context, B = h->cfg.hot_slots;
  const size_t r = req;
  cudaError_t e;
  if ((e = cudaMemsetAsync(h->s.page + r * L * N, 0xff, L * N * 4, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->s.reverse + r * L * B, 0xff, L * B * 4, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->s.stamp + r * L * B, 0xff, L * B * 4, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->s.length + r * L, 0, L * 4, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->s.step + r * L, 0, L * 4, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->s.hits + r * L, 0, L * 8, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->s.misses + r * L, 0, L * 8, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->s.cand_thr + r * L, 0, L * 4, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->s.sh_armed + r * L, 0, L * 4, st)) != cudaSuccess ||
      (e = hs::launch_init_order(h->s.order + r * L * B, (long long)L, (int)B, st)) != cudaSuccess)
    return cuda_fail(h, e, "hs_reset_request");
  return HS_OK;
}

int hs_set_timing(hs_handle_t* h, int32_t enable) {
  if (!h) return HS_ERR_INVALID;
  cudaSetDevice(h->cfg.device);
  cudaDeviceSynchronize();
  for (auto& t : h->timed) {
    h->event_pool.push_back(t.a);
    h->event_pool.push_back(t.b);
  }
  h->timed.clear();
  h->timing = enable != 0;
  return HS_OK;
}

int hs_kernel_times(hs_handle_t* h, double* ms, int64_t* launches) {
  if (!h || !ms || !launches) return HS_ERR_INVALID;
  cudaSetDevice(h->cfg.device);
  for (int k = 0; k < HS_K_COUNT; ++k) {
    ms[k] = 0.0;
    launches[k] = 0;
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e, "hs_kernel_times: synchronize");
  for (auto& t : h->timed) {
    float x = 0.f;
    if (cudaEventElapsedTime(&x, t.a, t.b) == cudaSuccess) {
      ms[t.kind] += x;
      launches[t.kind] += 1;
    }
  }
  (void)cudaGetLastError();
  return HS_OK;
}

}  // extern "C"
