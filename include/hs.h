/*
 * hs.h — C ABI of a two-level KV cache for top-k sparse-attention decode
 * (HiSparse), written for one NVIDIA GB300 GPU (sm_103a).
 *
 * What the library does, and where the method is stated:
 *   "KV卸载上主机:HiSparse、PDD与DDR4回收" (yeyulingfeng.com), section
 *   "二、论文分析 / 论文1：HiSparse": the authoritative full KV of every active
 *   request lives in pinned host DRAM; the GPU keeps a fixed hot cache of B slots
 *   per request per layer; a page table plus LRU metadata drive replacement; hit
 *   detection, LRU replacement, metadata update and the host fetch are fused into
 *   one RESOLVE kernel launched once per layer; only placement changes, so the
 *   attention result is exactly top-k sparse attention over the full KV.
 *   "10月14日学习笔记" (zgchen.com), section "HiSparse": the indexer picks the
 *   top-k tokens ("动机"); adjacent steps overlap and LRU fits them ("方法" 1);
 *   the whole flow runs without host involvement inside a CUDA graph ("方法" 2).
 *
 * Conventions for every call below:
 *   - Return value: HS_OK (0) or a negative HS_ERR_* status.  On error nothing
 *     was enqueued unless stated; hs_last_error() gives a message.
 *   - "dev" pointers are CUDA device pointers (or any address the GPU can
 *     dereference, e.g. pinned host memory under unified addressing); they stay
 *     owned by the caller and must stay valid until the enqueued work finishes.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls on one handle must be ordered on one stream (they share scratch).
 *   - bf16 tensors are raw bf16 bit patterns, row-major, densely packed.
 *   - Errors that only the GPU can see (a request id out of range, an append past
 *     max_context, a decode of an empty request, a bounded wait that gave up)
 *     do not fail the call: the kernel skips the affected request, sets a bit in
 *     the handle's device error word (HS_DEVERR_*), and hs_stats() reports it.
 */
#ifndef HS_H_
#define HS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define HS_OK 0
#define HS_ERR_INVALID (-1)  /* bad argument (null pointer, range, layer, count) */
#define HS_ERR_CONFIG (-2)   /* configuration outside what the kernels support */
#define HS_ERR_OOM (-3)      /* host or device allocation failed (all freed again) */
#define HS_ERR_CAPACITY (-4) /* request/position capacity exceeded (host-side check) */
#define HS_ERR_CUDA (-5)     /* a CUDA runtime call failed (message has the name) */
#define HS_ERR_DEVICE (-6)   /* hs_stats: the device error word is non-zero */

/* ---- bits of the device error word -------------------------------------- */
#define HS_DEVERR_REQ_RANGE 0x1u  /* a request id outside [0, max_requests) */
#define HS_DEVERR_CAPACITY 0x2u   /* append past max_context: request skipped, nothing written */
#define HS_DEVERR_EMPTY 0x4u      /* decode of a request with no positions: output set to 0 */
#define HS_DEVERR_TIMEOUT 0x8u    /* a bounded wait inside a kernel gave up */
#define HS_DEVERR_METADATA 0x10u  /* page table / reverse map found inconsistent */
#define HS_DEVERR_NO_LEAD 0x20u   /* a follower layer of a shared selection was decoded without
                                     its group lead's selection of the same step: output 0 */

/*
 * Configuration.  Positions and rows:
 *   A "row" is one position's K and V for all kv heads of one layer, bf16:
 *     GQA (shared_kv = 0): [K: h_kv x d_qk][V: h_kv x d_v], row_elems = h_kv*(d_qk+d_v)
 *     latent (shared_kv = 1, h_kv = 1): one row of d_qk elements read as K; its
 *       first d_v elements are V (DeepSeek-style MLA latent), row_elems = d_qk.
 *   q head h reads kv head floor(h * h_kv / h_q).
 * Supported by the kernels (else HS_ERR_CONFIG):
 *   GQA: d_qk = d_v = 128, h_q % h_kv == 0, h_kv in {1,2,4,8}, h_q/h_kv <= 16.
 *   latent: h_kv = 1, d_qk = 576, d_v = 512, h_q in {16, 32, 64, 128}.
 *   d_idx in {16, 32, 64, 128, 256}; 1 <= top_k <= hot_slots <= 16384, hot_slots % 4 == 0;
 *   top_k <= 8192; 1 <= max_context <= HS_MAX_CONTEXT; n_layers >= 1;
 *   1 <= max_requests <= 4096 (and every kernel's shared-memory layout must fit,
 *   else HS_ERR_CONFIG names the kernel).
 */
#define HS_MAX_CONTEXT (1 << 20)

typedef struct hs_config {
  int32_t n_layers;
  int32_t max_requests;  /* request ids are 0 .. max_requests-1 */
  int32_t max_context;   /* positions per (request, layer) */
  int32_t h_q;
  int32_t h_kv;
  int32_t d_qk;
  int32_t d_v;
  int32_t shared_kv;     /* 0: GQA rows, 1: latent rows (see above) */
  int32_t d_idx;         /* int8 index-key width */
  int32_t top_k;         /* k: positions attended per step */
  int32_t hot_slots;     /* B: HBM slots per (request, layer) */
  float softmax_scale;   /* 0 => 1/sqrt(d_qk) */
  int32_t device;        /* CUDA device ordinal */
  int32_t fetch_mode;    /* where missed rows are copied host -> HBM (results identical):
                            0 = by the loader warp of the attention kernel, into its stage
                                and from there into the slot, overlapping the HBM reads of
                                the hit rows;
                            1 = by RESOLVE (inside the select kernel), before the request
                                is handed to the attention kernel;
                            2 = the default: as 0.
                            RESOLVE starts every missed row moving into L2 as soon as
                            it finds it, whichever copies it.
                            Latent rows (shared_kv = 1) always use 1: every head
                            group reads them, so they cross the host link once. */
  int32_t replacement;   /* which unpinned slots the misses replace (hits are always pinned;
                            victims are the m unpinned slots with the smallest (stamp, slot)):
                            HS_REPLACE_LRU  (0): every slot the call uses (hits and fills)
                                gets stamp = step — least recently used first, the pages'
                                policy;
                            HS_REPLACE_FIFO (1): only filled slots get stamp = step, a hit
                                keeps its fill stamp — first filled first, the comparison
                                policy of the pages' miss-rate ablation;
                            HS_REPLACE_RANDOM (2): the other comparison policy: never-filled
                                unpinned slots go first (lowest first), the rest of the
                                victims are the unpinned filled slots with the smallest
                                (key, slot), key = the top 23 bits of SplitMix64 (Steele,
                                Lea and Flood 2014; Vigna's constants) at counter
                                ((request * n_layers + layer) << 40 | (step mod 2^24) << 16
                                | slot) + 1 from state replacement_seed, i.e.
                                z = replacement_seed + (counter + 1) * 0x9E3779B97F4A7C15,
                                z = (z ^ z >> 30) * 0xBF58476D1CE4E5B9,
                                z = (z ^ z >> 27) * 0x94D049BB133111EB, z ^= z >> 31,
                                key = z >> 41 (all mod 2^64): a uniformly random subset;
                                the victims are filled in ascending slot order; stamps as
                                for LRU.
                            The attention result does not depend on it. */
  uint32_t replacement_seed;  /* seed of HS_REPLACE_RANDOM (ignored otherwise) */
  int32_t write_allocate;     /* 0 (write-around, the default): an appended token enters the hot
                                 cache only when a later step selects it.  1: the token a
                                 hs_decode_layer call appends (new_kv_rows) counts as used by that
                                 call: when its selection does not take it, it is filled from its
                                 input row into one more victim slot (the last, after the
                                 selection's misses) and stamped like the rest; hits and misses
                                 still count the selected positions only.  Requires
                                 top_k < hot_slots.  Tokens appended by hs_append are never
                                 allocated.  The attention result does not depend on it. */
  int32_t idx_heads;          /* the indexer: 0 or 1 = one int8 query per request, score
                                 s[p] = q . K_idx[p] (signed, exact int32); 2, 4 or 8 = the
                                 multi-head ReLU-weighted variant (needs d_idx 64 or 128):
                                 s[p] = sum_h w_h * max(0, q_h . K_idx[p]), exact in uint32, with
                                 per-request query heads q_h and weights w_h in [0, 127]
                                 (negative weights count as 0).  Selection, ties and the cache
                                 rule are the same; the top-k then takes three digit passes over
                                 the keys and no candidate list. */
  int32_t index_share;        /* layers per indexer group, G (0 or 1: every layer selects for itself).
                                 With G > 1 (GQA rows only), layer l selects only when l % G == 0
                                 (the group's lead); layers l+1 .. l+G-1 of the same step reuse its
                                 selection, as a model that shares one indexer's choice across a
                                 group of layers does.  Every call of such a handle must append its
                                 token through new_kv_rows / new_idx_keys, and a step must call the
                                 lead before its followers (else HS_DEVERR_NO_LEAD, output 0). */
  int32_t share_prefetch;     /* with G > 1: 1 = the lead's call also resolves every follower layer
                                 (page table, LRU, stamps) and pulls its missed rows into its slots
                                 right away, so a follower's call only appends its token and attends
                                 (the prefetch that a shared selection makes exact); 0 = each
                                 follower resolves and pulls at its own call. */
  int32_t page_size;          /* 0 or 1: positions are selected and cached one by one.  P in
                                 {2, 4, 8, 16, 32, 64}: Quest-style page selection (GQA rows only).
                                 Positions form pages of P (page j = positions jP .. jP+P-1); each
                                 page keeps the element-wise maximum and minimum of its index keys
                                 (the page-bound store, [max_requests][n_layers][ceil(max_context/P)]
                                 [2 * d_idx] int8: maxima then minima, kept current by hs_append and
                                 by the appending decode call); a page scores
                                 U = sum_d max(q_d * kmax_d, q_d * kmin_d), the largest q . k any key
                                 within those bounds reaches (exact int32); the top_k / P pages with
                                 the largest U (ties: the lower page) are selected and every position
                                 of them below the length is attended (the selection output lists
                                 those positions ascending, then -1).  The hot cache then holds
                                 hot_slots / P page slots of P consecutive rows, and the page table,
                                 reverse map, stamps, LRU order and the hit / miss counters are per
                                 page and page slot (hs_snapshot: page[j] = page slot of page j;
                                 reverse, stamp and order: their first hot_slots / P entries).
                                 Requires top_k % P == 0, hot_slots % (4 P) == 0, d_idx 64 or 128,
                                 idx_heads <= 1, index_share <= 1 and write_allocate = 0. */
} hs_config_t;

#define HS_REPLACE_LRU 0
#define HS_REPLACE_FIFO 1
#define HS_REPLACE_RANDOM 2

typedef struct hs_handle hs_handle_t;

typedef struct hs_stats {
  uint64_t hits;          /* selected positions (pages, with page_size > 1) found in the hot cache */
  uint64_t misses;        /* selected positions (pages) pulled from host memory */
  uint64_t h2d_bytes;     /* bytes pulled host -> HBM by RESOLVE */
  uint64_t d2h_bytes;     /* K/V bytes written to the host copy by appends */
  uint64_t decode_calls;  /* hs_decode_layer calls enqueued */
  uint64_t append_calls;  /* hs_append calls enqueued */
  uint64_t host_bytes;    /* size of the pinned host K/V store */
  uint64_t hot_bytes;     /* size of the HBM hot cache */
  uint64_t index_bytes;   /* size of the HBM index-key store (with the page-bound store) */
  uint64_t meta_bytes;    /* page table, reverse map, stamps, LRU order, counters */
  uint64_t host_huge_bytes;  /* bytes of the host store backed by transparent huge pages when it
                                was created (random row reads over the link take about half as
                                long on them as on base pages) */
  uint64_t full_selects;  /* selections that scanned every key (no usable candidate list:
                             first steps, a large drift, contexts above 20 k positions) */
  /* Timing of the GQA attention kernel, from the device's global timer (latent-row
     calls add nothing).  One consumer warp per CTA times its waits for each stage
     of rows: stages holding at least one row read from host memory count as
     "host", the others as "hbm"; the difference of their mean waits is the host
     link's exposed latency per host stage. */
  uint64_t att_host_wait_ns;  /* summed over CTAs and calls: waits for host stages */
  uint64_t att_host_stages;   /* host stages waited for */
  uint64_t att_hbm_wait_ns;   /* summed over CTAs and calls: waits for hbm stages */
  uint64_t att_hbm_stages;    /* hbm stages waited for */
  uint64_t att_last_span_ns;  /* the latest GQA attention launch: its last CTA's end minus
                                 its first CTA's start (0 before the first launch) */
  uint64_t att_last_median_ns;  /* the same launch: the median CTA end minus the first
                                   CTA's start (load balance: span / median) */
  uint32_t device_error;  /* HS_DEVERR_* bits seen so far (sticky) */
  uint32_t _pad;
} hs_stats_t;

/*
 * hs_create — validate `cfg` and allocate every store (synchronous).
 *   host store  D1: [max_requests][n_layers][max_context][row] bf16, pinned and
 *                   mapped host memory: anonymous memory in whole transparent huge
 *                   pages (advised, faulted in, and what the kernel backed with
 *                   base pages collapsed with MADV_COLLAPSE; the coverage is in
 *                   hs_stats.host_huge_bytes), registered with cudaHostRegister
 *                   (Mapped | Portable), else cudaHostAlloc(Mapped | Portable):
 *                   the authoritative copy;
 *   hot cache   D2: [max_requests][n_layers][hot_slots][row] bf16 in HBM;
 *   index keys  D3: [max_requests][n_layers][max_context][d_idx] int8 in HBM;
 *   page table  D4: [max_requests][n_layers][max_context] int32, -1 = not resident;
 *   reverse map, stamps, (stamp, slot) order: [max_requests][n_layers][hot_slots]
 *   int32; per-(request, layer) length, step counter, hit and miss counters.
 *   All requests start empty (length 0, every slot empty, step 0).
 * Returns HS_ERR_INVALID (null), HS_ERR_CONFIG (unsupported shape), HS_ERR_OOM
 * (allocation failed; nothing stays allocated) or HS_ERR_CUDA.  On success
 * *out owns everything until hs_destroy.  The environment variable
 * HS_FAULT_INJECT=hostalloc|devalloc makes the first host / device allocation
 * fail (to test the clean-up path); HS_FAULT_INJECT=noready (read here) makes
 * every hs_decode_layer of the handle withhold the publication of its first
 * request, so the attention kernel's bounded wait for it runs out (after about
 * a second): the call sets HS_DEVERR_TIMEOUT, that request's output is
 * undefined, and the handle must be destroyed (to test the timeout path).
 */
int hs_create(const hs_config_t* cfg, hs_handle_t** out);

/* hs_destroy — synchronise the device and free everything; NULL is a no-op. */
void hs_destroy(hs_handle_t* h);

/*
 * hs_append — append n_tok tokens to each of n_req requests of one layer
 * (stream-ordered, no host synchronisation).
 *   req_ids : dev int32 [n_req] distinct request ids, or NULL for 0..n_req-1
 *   kv_rows : dev bf16 [n_req][n_tok][row_elems]   (device or pinned host memory)
 *   idx_keys: dev int8 [n_req][n_tok][d_idx]
 * For request r with current length L the tokens take positions L..L+n_tok-1:
 * their index keys go to the HBM key store, their K/V rows to the pinned host
 * copy (not to the hot cache: a new token enters the cache only when a later
 * step selects it), and the length becomes L+n_tok.  With page_size P > 1 the
 * bounds of every page the tokens touch are recomputed from the key store, and
 * a token whose page is resident in the hot cache also has its row written into
 * that page's slot (a page can be cached before all of its positions exist).
 * A request whose append
 * would pass max_context is skipped whole (HS_DEVERR_CAPACITY).
 * n_req = 0 or n_tok = 0 is a no-op.  HS_ERR_INVALID for layer out of range,
 * n_req > max_requests, n_tok > max_context or a null buffer.
 */
int hs_append(hs_handle_t* h, int32_t layer, int32_t n_req, const int32_t* req_ids,
              int32_t n_tok, const void* kv_rows, const int8_t* idx_keys, void* stream);

/*
 * hs_decode_layer — one decode layer-step for n_req requests (stream-ordered,
 * no host synchronisation, capturable in a CUDA graph).  Two kernels: the select
 * kernel (scores, top-k, RESOLVE) waits for the previous kernel of the stream
 * before it reads anything; the attention kernel is launched as its
 * programmatic dependent and starts on each request as soon as that request is
 * resolved, and completes only after the select kernel has.  So ordering against
 * earlier and later stream work is the usual one.  At most 32 requests are
 * resolved at a time (one resolver CTA each); the rest of the GPU scores.
 *   req_ids     : dev int32 [n_req] distinct request ids, or NULL for 0..n_req-1
 *   q_idx       : dev int8 [n_req][d_idx]       indexer query (16-byte aligned); with
 *                 idx_heads = H > 1: [n_req][H * d_idx + 16], per request the H query
 *                 heads, then the H weights (int8), then padding
 *   q           : dev bf16 [n_req][h_q][d_qk]   attention query
 *   out         : dev bf16 [n_req][h_q][d_v]    attention output (written)
 *   sel_out     : dev int32 [n_req][top_k] or NULL: selected positions, ascending;
 *                 entries past k_eff = min(top_k, length) are -1
 *   new_kv_rows : dev bf16 [n_req][row_elems] or NULL (16-byte aligned)
 *   new_idx_keys: dev int8 [n_req][d_idx] or NULL (both or neither)
 * With new_kv_rows / new_idx_keys the call first appends one token per request,
 * exactly as hs_append with n_tok = 1 would (same positions, stores and length
 * update; a request at max_context gets HS_DEVERR_CAPACITY and no append), but
 * inside the decode kernels instead of a launch of its own.
 * Per request with N positions: (1) score every position p < N as
 * sum_j q_idx[j] * K_idx[p][j] (exact int32); (2) keep the k_eff highest, ties
 * to the lower position; (3) RESOLVE: hits via the page table, misses assigned to
 * victim slots of the configured replacement policy (LRU unless set otherwise),
 * metadata and stamps updated, step += 1, missed rows copied
 * from the host copy into their slots (by RESOLVE or by the attention kernel,
 * see fetch_mode); (4) o_h = sum_i softmax_i(scale * q_h . K_i) V_i over the
 * selected rows in ascending position order, fp32 accumulation, bf16 output.
 * The output does not depend on hot_slots or on the cache state (bit-identical
 * across B).  HS_ERR_INVALID for layer out of range, n_req > max_requests, null or
 * misaligned buffers.
 */
int hs_decode_layer(hs_handle_t* h, int32_t layer, int32_t n_req, const int32_t* req_ids,
                    const int8_t* q_idx, const void* q, void* out, int32_t* sel_out,
                    const void* new_kv_rows, const int8_t* new_idx_keys, void* stream);

/*
 * hs_stats — synchronise the device and fill *out with cumulative counters and
 * sizes.  Returns HS_ERR_DEVICE (with *out filled) when the device error word is
 * non-zero, HS_ERR_INVALID for null arguments.
 */
int hs_stats(hs_handle_t* h, hs_stats_t* out);

/*
 * hs_snapshot — synchronise and copy the cache state of one (request, layer)
 * to host buffers (test and debugging introspection).  Any output may be NULL.
 *   page    : int32 [n_page]   page-table entries of positions 0..n_page-1
 *   reverse : int32 [hot_slots] position held by each slot, -1 = empty
 *   stamp   : int32 [hot_slots] step of last use of each slot (FIFO: of its last
 *             fill), -1 = never
 *   order   : int32 [hot_slots] slots from least to most recently used
 *             (sorted by (stamp, slot))
 *   scalars : int64 [4] = {length, step, hits, misses} of this (request, layer)
 * HS_ERR_INVALID for out-of-range req/layer or n_page > max_context.
 */
int hs_snapshot(hs_handle_t* h, int32_t req, int32_t layer, int32_t* page, int32_t n_page,
                int32_t* reverse, int32_t* stamp, int32_t* order, int64_t* scalars);

/*
 * hs_reset_request — forget request `req` on every layer (stream-ordered):
 * length 0, page table cleared, every slot empty, step 0, counters 0.  Used to
 * recycle a request id.  HS_ERR_INVALID when req is out of range.
 */
int hs_reset_request(hs_handle_t* h, int32_t req, void* stream);

/*
 * hs_set_timing / hs_kernel_times — per-kernel device timing.  With timing on,
 * every launch is bracketed by CUDA events on the caller's stream (so the
 * attention kernel no longer starts while the select kernel still runs: the
 * times are those of each kernel alone); hs_kernel_times
 * synchronises and returns, per kernel kind (HS_K_*), the summed milliseconds and
 * the number of launches since the last hs_set_timing(h, 1).
 */
#define HS_K_APPEND 0     /* append kernel (hs_append) */
#define HS_K_SELECT 1     /* the select kernel of hs_decode_layer: scores, exact top-k and RESOLVE
                             (and the host fetch when fetch_mode = 1 or rows are latent) */
#define HS_K_ATTENTION 2  /* the attention kernel, which also merges its partials (and does the
                             host fetch when fetch_mode = 0 or 2); latent rows: attention +
                             merge kernels */
#define HS_K_COUNT 3
int hs_set_timing(hs_handle_t* h, int32_t enable);
int hs_kernel_times(hs_handle_t* h, double* ms /*[HS_K_COUNT]*/, int64_t* launches /*[HS_K_COUNT]*/);

/*
 * hs_indexer_topk_static — the indexer scores and exact top-k selection of
 * hs_decode_layer (its steps 1 and 2, without the cache update) for callers
 * that cannot allocate device memory: code that runs where cudaMalloc is not
 * available or not allowed, such as inside another allocator's critical section,
 * under a memory pool that forbids side allocations, or in a plugin that is only
 * handed raw buffers.  The pages have no counterpart to this entry point.
 * It allocates nothing (no cudaMalloc, cudaFree or allocating library call).  Its
 * scratch — 64 histograms of 4096 bins and up to 2^21 32-bit keys, about 9 MiB —
 * is one file-scope device array, which every GPU that loads the library holds
 * until the process exits.
 *   n_req    : requests, 0..64 (more: HS_ERR_CAPACITY)
 *   n_max    : positions stride of idx_keys; n_req * round_up(n_max, 4) <= 2^21
 *              (more: HS_ERR_CAPACITY)
 *   d_idx    : 16, 32, 64, 128 or 256;   top_k : k >= 1
 *   idx_keys : dev int8 [n_req][n_max][d_idx], 16-byte aligned
 *   lengths  : HOST int32 [n_req], each in [0, n_max]: positions of each request
 *   q_idx    : dev int8 [n_req][d_idx], 16-byte aligned
 *   sel_out  : dev int32 [n_req][top_k]: the k_eff = min(top_k, length) highest
 *              scores' positions, ascending, ties to the lower position, then -1
 *              (the same values hs_decode_layer writes to its sel_out)
 *   device   : CUDA device to run on (made current);  stream : cudaStream_t as void*
 * The first call on a device does a one-time set-up with that device current (it
 * looks up the device address of the array); make that first call before any
 * stream capture.  All calls on a device share the array, which keeps the last
 * call's contents: calls that overlap on the GPU (different streams, concurrent
 * replays) race and must be ordered by the caller.  A non-zero status comes with
 * a message in hs_last_error(NULL).  Errors only the GPU can see (a bounded wait
 * inside the score kernel that gave up) make the call write -1 to every entry
 * of sel_out and set the device error word that hs_indexer_topk_static_error
 * reads.
 */
int hs_indexer_topk_static(int32_t n_req, int32_t n_max, int32_t d_idx, int32_t top_k,
                           const int8_t* idx_keys, const int32_t* lengths, const int8_t* q_idx,
                           int32_t* sel_out, int32_t device, void* stream);

/*
 * hs_indexer_topk_static_error — synchronise `device` and read the device error
 * word (HS_DEVERR_* bits) left by the most recent hs_indexer_topk_static call on
 * it (each call clears the word first).  *out = 0 and HS_OK when no call has run
 * on the device; HS_ERR_DEVICE (with *out set) when the word is non-zero;
 * HS_ERR_INVALID for a null `out` or a device out of range.  Allocates nothing.
 */
int hs_indexer_topk_static_error(int32_t device, uint32_t* out);

/* hs_last_error — message of the handle's last failed call ("" if none); with
 * h == NULL, the message of the last failed hs_create in this thread. */
const char* hs_last_error(const hs_handle_t* h);

/* hs_status_string — static name of a status code. */
const char* hs_status_string(int32_t status);

/* hs_row_elems — bf16 elements of one K/V row under cfg (0 if cfg is invalid). */
int32_t hs_row_elems(const hs_config_t* cfg);

#ifdef __cplusplus
}
#endif

#endif /* HS_H_ */
