// Internal declarations shared by the CUDA translation units of the library:
// the handle, the per-kernel parameter blocks, launch helpers and small
// device-side primitives (PTX wrappers for mbarriers and bulk copies, block scans).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "hs.h"

namespace hs {

constexpr unsigned FULL_MASK = 0xffffffffu;

// ---- geometry fixed by the kernels ------------------------------------------
constexpr int SC_THREADS = 256;      // score kernel CTA
constexpr int IDX_TILE_BYTES = 32768;  // index keys per bulk copy (one tile)
constexpr int IDX_BINS = 4096;       // radix digit: 12 bits, two levels cover 24-bit keys
constexpr int IDX_KEY_BIAS = 1 << 22;  // |score| <= 128*128*256 = 2^22 for d_idx <= 256

constexpr int RES_THREADS = 1024;    // top-k CTA of the static (no-allocation) entry point

// The select kernel (scores, top-k and RESOLVE in one persistent launch): every
// CTA has SEL_THREADS threads; a scorer CTA runs two independent 256-thread
// scoring groups, a resolver CTA runs the top-k + RESOLVE chain of its requests.
constexpr int SEL_THREADS = 512;
constexpr int SEL_GROUP = 256;       // threads of one scoring group
constexpr int SEL_MAX_RESOLVERS = 32;
constexpr int ROLE_SELECT = 0, ROLE_GIVEN = 1;

// slot_of_sel entries of rows RESOLVE left for the attention kernel to fetch
constexpr int HS_SLOT_MISS_FLAG = 0x40000000;

constexpr int ATT_SUBTILE = 16;      // rows per warp per tile
constexpr int ATT_ROW_PAD = 16;      // bytes of padding per row in shared memory (bank spread)

constexpr int APP_THREADS = 256;
constexpr int APP_TOKENS_PER_CTA = 16;

// one bounded wait gives up after this many nanoseconds of wall time
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;

// ---- parameter blocks -------------------------------------------------------
struct Geometry {
  int n_layers, max_requests, max_context;
  int h_q, h_kv, d_qk, d_v, shared_kv, d_idx, top_k, hot_slots;
  int row_elems, row_bytes, v_off;
  int idx_heads;           // 1: one indexer query (signed score); 2/4/8: the multi-head ReLU-weighted indexer
  int page_size;           // 1: positions are selected and cached one by one; P > 1: pages of P positions
  int page_shift;          // log2(page_size)
  int max_pages;           // pages per (request, layer): ceil(max_context / page_size)
};

struct DeviceState {
  uint16_t* host_kv;       // device alias of the pinned host store [R][L][Nmax][row]
  uint16_t* hot;           // [R][L][B][row]
  int8_t* idx_keys;        // [R][L][Nmax][d_idx]
  int8_t* pbound;          // [R][L][max_pages][2 * d_idx] page mode: per page [max | min] of its keys
  int32_t* page;           // [R][L][Nmax]
  int32_t* reverse;        // [R][L][B]
  int32_t* stamp;          // [R][L][B]
  int32_t* order;          // [R][L][B]  slots by (stamp, slot) ascending
  int32_t* length;         // [R][L]
  int32_t* step;           // [R][L]
  unsigned long long* hits;    // [R][L]
  unsigned long long* misses;  // [R][L]
  unsigned long long* glob;    // [0] h2d bytes, [1] d2h bytes, [2] selections over every key,
                               // [4..7] attention stage waits: host ns, host stages, hbm ns, hbm stages
  unsigned long long* att_cta;  // [att_grid][2] (start, end) global-timer ns of each attention CTA, latest launch
  unsigned int* dev_error;     // sticky HS_DEVERR_* bits
  // scratch (one call in flight per handle)
  uint32_t* scores;        // [R][score_stride] 24-bit keys of the current call
  uint32_t* hist;          // [R][4096] high-digit histogram of the current call (zero between calls)
  // candidate pre-filter: keys at or above the (request, layer)'s threshold from
  // the previous call, listed by the score kernel for the top-k
  uint32_t* cand_thr;      // [R][L] threshold for the next call (0: none)
  uint32_t* cand_cnt;      // [R] keys listed in the current call (zero between calls)
  uint2* cand;             // [R][2k] (position, key), unordered
  int32_t* cand_slot;      // [R][2k] page-table entry of each listed unit, read by the scorer that lists it
  int32_t* sel;            // [R][k]
  int32_t* slot_of_sel;    // [R][k]
  float* part_o;           // [R][parts][h_q][d_v]
  float* part_ml;          // [R][parts][h_q][2]
  int32_t* att_nparts;     // [R][8] partial results of each (request, head group) of the current call
  int32_t* call_n;         // [R] positions of request i in the current call (with its appended token)
  unsigned int* app_counter;   // [R]
  // cross-CTA progress of one decode call (all zero between calls: every counter
  // is reset by the last party that reads it)
  unsigned int* tiles_done;    // [R] score tiles of request i finished (select kernel)
  unsigned int* ready;         // [R] k_eff + 1 once request i's selection and slots are published
  // the units request i misses this call, listed by RESOLVE as soon as they are
  // known (before publication) for the attention kernel's host-row prefetch: a
  // hint only (written and read without ordering; every entry is bounds-checked)
  unsigned int* miss_cnt;      // [R] misses listed + 1 (0: not yet)
  unsigned int* att_done;      // [R] chunks of request i whose partials the attention kernel has written
  int32_t* miss_pos;           // [R][k] unit index of each listed miss
  // a selection shared by a group of layers (index_share > 1): what the group's
  // lead call leaves for each follower layer [R][L][...]
  int32_t* sh_sel;             // [R][L][k] the shared selection (positions, ascending)
  int32_t* sh_slots;           // [R][L][k] the follower's slot of each (resolved ahead)
  int32_t* sh_kk;              // [R][L] k_eff
  int32_t* sh_pend;            // [R][L] slot awaiting the follower's own appended row (-1: none)
  int32_t* sh_armed;           // [R][L] 1: left by the lead of this step, not yet used
  unsigned int* sync;          // [8]: 0 = CTAs of the select kernel past their set-up,
                               //      1 = resolvers finished, 2 = next attention work item,
                               //      3 = attention CTAs finished, 4 = next request whose
                               //      missed rows the attention kernel prefetches, 5 = next
                               //      merge item of the attention kernel
};

struct AppendParams {
  Geometry g;
  DeviceState s;
  int layer, n_req, n_tok;
  const int32_t* req_ids;
  const uint16_t* kv_rows;
  const int8_t* keys;
};

struct DecodeParams {
  Geometry g;
  DeviceState s;
  int layer, n_req;
  const int32_t* req_ids;
  const int8_t* q_idx;
  const uint16_t* q;
  uint16_t* out;
  int32_t* sel_out;
  const uint16_t* new_kv;  // [n_req][row] token appended by this call, or null
  const int8_t* new_keys;  // [n_req][d_idx]
  float scale_log2;        // softmax scale * log2(e)
  long long score_stride;  // scores row stride (positions, multiple of 4)
  int score_grid;          // score kernel CTAs
  int att_parts;           // partial results per request (CTAs x slices)
  int att_grid;            // attention CTAs (one per SM)
  int fetch_mode;          // 0: attention kernel fetches misses, 1: RESOLVE does
  int replacement;         // HS_REPLACE_LRU / _FIFO / _RANDOM
  unsigned int replacement_seed;
  int sel_grid;            // select kernel CTAs (one per SM)
  int n_resolvers;         // of them, resolver CTAs (the rest score)
  int publish;             // 1: resolvers publish each request (the chunked attention kernel waits on it)
  int fault;               // test hook: 1 = the resolver never publishes request 0 (a wait runs out)
  int write_allocate;      // 1: the token this call appends counts as used (filled if not selected)
  int role;                // ROLE_SELECT: this call selects; ROLE_GIVEN: it resolves the selection its
                           // group's lead left (no scoring)
  int n_follow;            // ROLE_SELECT with index_share: follower layers of the group after this one
  int share_prefetch;      // 1: resolve the followers now (pulling their missed rows ahead); 0: leave
                           // the selection for them to resolve at their own calls
#ifdef HS_WITH_TRACE
  unsigned long long* trace;   // [2][3][1024][64]: clock64 and %globaltimer per (kernel, CTA, point)
#endif
};

}  // namespace hs

// ---- the handle -----------------------------------------------------------------
struct hs_handle {
  hs_config_t cfg;
  hs::Geometry g;
  hs::DeviceState s;
  uint16_t* host_kv_host = nullptr;   // host view of the pinned store
  void* host_map_base = nullptr;      // the store's mapping when it was registered (else cudaHostAlloc)
  size_t host_map_bytes = 0;
  size_t host_huge_bytes = 0;        // of the store, backed by transparent huge pages at create
  float scale_log2 = 0.f;
  int num_sms = 0;
  long long score_stride = 0;
  size_t sel_smem = 0, att_smem = 0;
  int fault = 0;                       // HS_FAULT_INJECT=noready at create (test hook)
  int att_parts = 0;
  size_t host_bytes = 0, hot_bytes = 0, index_bytes = 0, meta_bytes = 0;
  uint64_t decode_calls = 0, append_calls = 0;
  std::vector<void*> dev_allocs;
  // timing
  bool timing = false;
  struct Timed { int kind; cudaEvent_t a, b; };
  std::vector<Timed> timed;
  std::vector<cudaEvent_t> event_pool;
  std::string last_error;
#ifdef HS_WITH_TRACE
  unsigned long long* trace = nullptr;
#endif
};

namespace hs {

// launchers (one per kernel translation unit); return a CUDA error code
cudaError_t launch_append(const AppendParams& p, cudaStream_t st);
cudaError_t launch_page_bounds(const AppendParams& p, cudaStream_t st);
cudaError_t launch_score(const DecodeParams& p, size_t smem, cudaStream_t st);
cudaError_t launch_select(const DecodeParams& p, size_t smem, cudaStream_t st);
cudaError_t launch_follow(const DecodeParams& p, cudaStream_t st);
size_t select_smem_bytes(const Geometry& g);
cudaError_t prepare_select(const Geometry& g, size_t smem);
cudaError_t launch_attention(const DecodeParams& p, size_t smem, cudaStream_t st);
cudaError_t launch_init_order(int32_t* order, long long n_lists, int B, cudaStream_t st);
// records a message for hs_last_error(NULL) and returns `code`
int set_static_error(int code, const char* msg);

// shared-memory needs, checked against the device limit at create time
size_t score_smem_bytes(const Geometry& g);
size_t attention_smem_bytes(const Geometry& g);
int attention_parts(const Geometry& g);
cudaError_t prepare_score(const Geometry& g, size_t smem);
cudaError_t prepare_attention(const Geometry& g, size_t smem);
// attention over shared latent rows (hs_attention_mla.cu) and the partial merge
int mla_parts(const Geometry& g);
size_t mla_smem_bytes(const Geometry& g);
cudaError_t dispatch_mla(const Geometry& g, const DecodeParams* p, size_t smem, cudaStream_t st);
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t st);

// Raises a kernel's dynamic shared-memory allowance to at least `smem`, never
// lowers it: several handles (of different shapes) share the kernels.  Every
// kernel of the decode path also prefers the largest shared-memory carveout, so
// consecutive kernels run with the same L1/shared split and the SMs need no
// reconfiguration between them.
template <typename F>
inline cudaError_t allow_smem(F* kern, size_t smem) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.preferredShmemCarveout != (int)cudaSharedmemCarveoutMaxShared) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  if ((size_t)fa.maxDynamicSharedSizeBytes >= smem) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// Launches a kernel that may start while the previous kernel in the stream is
// still finishing (programmatic dependent launch).  Every such kernel runs
// griddep_wait() before it reads anything earlier stream work wrote, and calls
// griddep_launch_dependents() only after that wait, so a kernel that starts
// early can rely on every kernel before its immediate predecessor having
// completed.  Shared-memory set-up and barrier initialisation overlap the
// predecessor's tail; in a CUDA graph the edge becomes a programmatic one.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---- device helpers -------------------------------------------------------------
#if defined(__CUDACC__)

// Waits until the preceding kernel of the stream has completed and its writes are
// visible (returns at once when the kernel was launched without the
// programmatic attribute).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel of the stream begin launching.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Phase timeline for performance work (builds with -DHS_WITH_TRACE only): the SM
// cycle counter and the global timer at point `pt` of kernel `k`, per CTA, for
// the latest launch.  Compiled out otherwise.
constexpr int TRACE_KERNELS = 3, TRACE_CTAS = 1024, TRACE_POINTS = 64;
#ifdef HS_WITH_TRACE
#define HS_TRACE_IF(p, k, pt, cond)                                                               \
  do {                                                                                            \
    if ((cond) && (p).trace && blockIdx.x < TRACE_CTAS) {                                         \
      const size_t i_ = ((size_t)(k) * TRACE_CTAS + blockIdx.x) * TRACE_POINTS + (pt);            \
      (p).trace[i_] = clock64();                                                                  \
      (p).trace[(size_t)TRACE_KERNELS * TRACE_CTAS * TRACE_POINTS + i_] = global_timer_ns();     \
    }                                                                                             \
  } while (0)
// a measured quantity (a summed wait in ns, a count) in place of a timestamp
#define HS_TRACE_VAL(p, k, pt, val)                                                               \
  do {                                                                                            \
    if ((p).trace && blockIdx.x < TRACE_CTAS) {                                                   \
      const size_t i_ = ((size_t)(k) * TRACE_CTAS + blockIdx.x) * TRACE_POINTS + (pt);            \
      (p).trace[i_] = 0;                                                                          \
      (p).trace[(size_t)TRACE_KERNELS * TRACE_CTAS * TRACE_POINTS + i_] = (val);                 \
    }                                                                                             \
  } while (0)
#define HS_TNOW() global_timer_ns()
#else
#define HS_TRACE_IF(p, k, pt, cond) \
  do {                              \
  } while (0)
#define HS_TRACE_VAL(p, k, pt, val) \
  do {                              \
  } while (0)
#define HS_TNOW() 0ull
#endif
#define HS_TRACE(p, k, pt) HS_TRACE_IF(p, k, pt, threadIdx.x == 0)

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity; gives up after WAIT_LIMIT_NS and
// returns false (the caller records HS_DEVERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
}

// Bulk (non-tensor) asynchronous copy global -> this CTA's shared memory,
// completing `bytes` transaction bytes on `bar`.  Both addresses 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16-byte LSU async copy global (device or mapped host memory) -> shared.
// L2 policy for data read once (streams): evicted first, so data that is
// reused soon (scores, partials, prefetched host rows) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Starts bringing `bytes` (a multiple of 16) at a 16-byte aligned global address
// into L2; a hint: no data returns and nothing waits on it.
// The 128-byte line holding `gsrc` towards L2 (no alignment needed).
__device__ __forceinline__ void prefetch_line_l2(const void* gsrc) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(gsrc));
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ int4 ld_nc_v4(const void* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void set_error(unsigned int* word, unsigned int bit) { atomicOr(word, bit); }

// byte-wise signed maximum / minimum of 16 int8 values (page key bounds)
__device__ __forceinline__ int4 vmax16(int4 a, int4 b) {
  return make_int4(__vmaxs4(a.x, b.x), __vmaxs4(a.y, b.y), __vmaxs4(a.z, b.z), __vmaxs4(a.w, b.w));
}
__device__ __forceinline__ int4 vmin16(int4 a, int4 b) {
  return make_int4(__vmins4(a.x, b.x), __vmins4(a.y, b.y), __vmins4(a.z, b.z), __vmins4(a.w, b.w));
}

// GPU-scope release add / store and acquire load: the publication of one CTA's
// writes to CTAs of the same or a concurrently running kernel.
__device__ __forceinline__ void red_release_add(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int atom_acq_rel_add(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_release(unsigned int* p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Spins until *p >= target (acquire), backing off from 32 ns to 512 ns between
// polls (many CTAs may poll one flag); gives up after limit_ns (WAIT_LIMIT_NS
// unless given) and returns false.
__device__ __forceinline__ bool wait_counter(const unsigned int* p, unsigned int target,
                                             unsigned long long limit_ns = WAIT_LIMIT_NS) {
  if (ld_acquire(p) >= target) return true;
  const unsigned long long t0 = global_timer_ns();
  unsigned ns = 32;
  for (uint32_t it = 1;; ++it) {
    __nanosleep(ns);
    if (ns < 512) ns <<= 1;
    if (ld_acquire(p) >= target) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}
// Named barrier over `n` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Fire-and-forget 64-bit add (no value returned, so the issuing thread never waits).
__device__ __forceinline__ void red_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// bf16 pair (low half = element 0) -> two floats
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Exclusive prefix sum of one value per thread over the block.  `scratch` holds
// NT/32 + 1 ints; every thread of the block must call it.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int x = lane < NW ? scratch[lane] : 0;
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(FULL_MASK, xi, o);
      if (lane >= o) xi += n;
    }
    if (lane < NW) scratch[lane] = xi - x;
    if (lane == NW - 1) scratch[NW] = xi;
  }
  __syncthreads();
  const int excl = incl - v + scratch[warp];
  if (total) *total = scratch[NW];
  __syncthreads();
  return excl;
}

// Two exclusive prefix sums at once (one set of barriers).  `scratch` holds
// 2 * (NT/32 + 1) ints.
template <int NT>
__device__ __forceinline__ int2 block_exclusive_scan2(int a, int b, int* scratch, int* tot_a, int* tot_b) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int na = __shfl_up_sync(FULL_MASK, ia, o);
    const int nb = __shfl_up_sync(FULL_MASK, ib, o);
    if (lane >= o) {
      ia += na;
      ib += nb;
    }
  }
  if (lane == 31) {
    scratch[warp] = ia;
    scratch[NW + 1 + warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    const int xa = lane < NW ? scratch[lane] : 0;
    const int xb = lane < NW ? scratch[NW + 1 + lane] : 0;
    int sa = xa, sb = xb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int na = __shfl_up_sync(FULL_MASK, sa, o);
      const int nb = __shfl_up_sync(FULL_MASK, sb, o);
      if (lane >= o) {
        sa += na;
        sb += nb;
      }
    }
    if (lane < NW) {
      scratch[lane] = sa - xa;
      scratch[NW + 1 + lane] = sb - xb;
    }
    if (lane == NW - 1) {
      scratch[NW] = sa;
      scratch[2 * NW + 1] = sb;
    }
  }
  __syncthreads();
  const int2 r = make_int2(ia - a + scratch[warp], ib - b + scratch[NW + 1 + warp]);
  if (tot_a) *tot_a = scratch[NW];
  if (tot_b) *tot_b = scratch[2 * NW + 1];
  __syncthreads();
  return r;
}

template <int NT>
__device__ __forceinline__ int block_sum(int v, int* scratch) {
  int total;
  block_exclusive_scan<NT>(v, scratch, &total);
  return total;
}

#endif  // __CUDACC__

}  // namespace hs
