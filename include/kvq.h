/*
 * kvq.h -- C ABI of the GB300 (sm_103a) mixed INT2/INT4 paged KV cache (with INT3
 * and FP4 pages as further widths) and its decode-step attention.
 *
 * The problem these calls follow:
 *   - TriAxialKV, key design 3 (custom mixed-precision cache layout and
 *     residual fallback): asymmetric group quantization with G = 32; INT4 K
 *     and V per token; INT2 K per channel with scale and zero shared across 32
 *     tokens; INT2 V per token; tokens that cannot fill a 32-token INT2 group
 *     stay INT4.
 *   - TriAxialKV, key design 4 (unified address space dual pool and fused
 *     Flash-Decoding): INT2 and INT4 pages live in one address range and a
 *     page's precision follows from its id; before decoding, each request's
 *     page table is reordered so INT2 pages precede INT4 pages; decoding splits
 *     the sequence, dequantizes inside the attention scan and merges the splits
 *     with a global log-sum-exp; new tokens are written as INT4 at the tail.
 *   - HyQuant, Algorithm 3 (decode): split-K over the quantized prefix with
 *     in-kernel dequantization, the g query heads of one KV head packed
 *     together, and a ReduceSoftmax merge of (m, l, acc).
 *   - IntentKV, method 2 (layout-preserving eviction): an evicted slot reads
 *     as a sentinel dead slot whose attention contribution is zero, and no
 *     surviving page moves.
 *
 * Conventions for every call:
 *   - Return value: a kv_status_t.  On KV_ERR_INVALID_ARG and KV_ERR_OOM the
 *     pool is left exactly as it was.  kv_last_error() gives a message for the
 *     calling thread's last failure.
 *   - "device" pointers are CUDA device memory on the pool's device, owned by
 *     the caller; "host" pointers are ordinary host memory owned by the caller
 *     and only read or written during the call.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously on it; device-side failures (an out-of-range
 *     input value found by the quantizer, a bounded wait that expired) are
 *     recorded in the pool and returned by kv_pool_sync().
 *   - A pool is not thread-safe; issue its calls from one thread and keep its
 *     device work on one stream at a time.
 *   - No C++ exception crosses this boundary.
 *
 * Fixed format: head_dim 128, 32 tokens per page, group size 32.  Page block
 * of one (page, kv head): INT2 = 3072 bytes, INT4 = 5120 bytes, INT3 = 4096
 * bytes, FP4 = 4608 bytes (codes plus binary16 scale/zero; FP4 scales only).
 * The physical byte order inside a block is private to the library;
 * kv_export_request() returns the canonical content.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = 1,     /* bad argument or size; nothing changed */
  KV_ERR_OOM = 2,             /* pool pages, table slots or request slots exhausted; nothing changed */
  KV_ERR_RANGE = 3,           /* an appended K/V value was NaN, Inf or |x| > 65504 */
  KV_ERR_CUDA = 4,            /* a CUDA runtime call failed */
  KV_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait gave up */
  KV_ERR_STATE = 6            /* call not valid in the pool's current state */
} kv_status_t;

typedef enum {
  KV_DECODE_AUTO = 0,         /* the fastest implementation available */
  KV_DECODE_SIMT = 1,         /* CUDA-core fp32 scan (reference/ablation kernel) */
  KV_DECODE_MMA = 2           /* tensor-core scan */
} kv_decode_impl_t;

typedef struct kv_pool kv_pool_t;   /* opaque; owns all pool device memory, tables and workspaces */

typedef struct {
  int32_t num_kv_heads;           /* Hkv >= 1 */
  int32_t head_dim;               /* must be 128 */
  int32_t page_tokens;            /* must be 32 */
  int32_t group;                  /* must be 32 */
  int64_t n_int2_pages;           /* INT2 page ids are [0, n_int2_pages) */
  int64_t n_int4_pages;           /* INT4 page ids are [n_int2_pages, n_int2_pages + n_int4_pages) */
  int32_t max_requests;           /* request ids are [0, max_requests) */
  int32_t max_pages_per_request;  /* table capacity of one request */
  int32_t device;                 /* CUDA device ordinal */
  int64_t n_int3_pages;           /* INT3 page ids are [n2 + n4, n2 + n4 + n_int3_pages); 0: none */
  int64_t n_fp4_pages;            /* FP4 (E2M1) page ids follow the INT3 ids; 0: none */
} kv_pool_config_t;

/* Width value of FP4 (E2M1) tokens in kv_append_quant's bits array. */
#define KV_WIDTH_FP4 0xF4

/* Create a pool: one device allocation holding the INT2 region followed by the
 * INT4 region (TriAxialKV key design 4) and, with n_int3_pages > 0, the INT3
 * region (TriAxialKV, limitations and outlook: INT3 as a further width; an
 * INT3 block is 4096 bytes per page and kv head) and, with n_fp4_pages > 0,
 * the FP4 region (the same section's non-uniform FP formats; 4608 bytes per
 * block), plus the device page tables.  out: host pointer receiving the
 * handle. */
KVQ_API kv_status_t kv_pool_create(const kv_pool_config_t* cfg, kv_pool_t** out);

/* Free everything the pool owns.  Synchronizes with the pool's device work. */
KVQ_API kv_status_t kv_pool_destroy(kv_pool_t* pool);

/* Open an empty request; *req_id (host) receives the lowest free request id. */
KVQ_API kv_status_t kv_request_open(kv_pool_t* pool, int32_t* req_id);

/* Close a request and return all of its pages to the free lists. */
KVQ_API kv_status_t kv_request_close(kv_pool_t* pool, int32_t req_id);

/* Quantize-on-append (TriAxialKV key designs 3 and 4).
 *   k, v     device, bf16 [n_tok][num_kv_heads][128], tokens in arrival order.
 *   req_ids  host, int32 [n_tok]: open request of each token.
 *   bits     host, uint8 [n_tok]: 4 -> the request's INT4 tail page;
 *            3 -> the request's INT3 tail page (K and V per token in groups of
 *            32 channels, codes 0..7, as INT4; needs n_int3_pages > 0);
 *            KV_WIDTH_FP4 -> the request's FP4 tail page (E2M1 values, K and V
 *            per token in groups of 32 channels with a binary16 scale
 *            max|x| / 6 and no zero point; the nearest value, ties to the even
 *            mantissa; needs n_fp4_pages > 0);
 *            2 -> the request's INT4 staging page, which is requantized into a
 *            new INT2 page (K per channel, V per token) as soon as it holds 32
 *            tokens; that INT2 page is appended to the request's table.
 * Page ids are the lowest free ids of their class; staging pages freed by a
 * repack become reusable after the call.  Values are checked on the device:
 * NaN, Inf or |x| > 65504 make kv_pool_sync() return KV_ERR_RANGE.  A request
 * holds at most 2^31 - 1 token positions: a call that would pass it returns
 * KV_ERR_INVALID_ARG with nothing changed; running out of pages or of the
 * request's table entries returns KV_ERR_OOM, also with nothing changed. */
KVQ_API kv_status_t kv_append_quant(kv_pool_t* pool, const void* k, const void* v, const int32_t* req_ids,
                            const uint8_t* bits, int64_t n_tok, void* stream);

/* Phase-1 reorder (TriAxialKV key design 4): stable partition of each listed
 * request's table so INT2 entries precede INT4 entries; with INT3 or FP4
 * pages, a stable sort by width (INT2, INT3, INT4, FP4).  req_ids: host [n_req]. */
KVQ_API kv_status_t kv_reorder_pages(kv_pool_t* pool, const int32_t* req_ids, int32_t n_req, void* stream);

/* Layout-preserving eviction (IntentKV method 2): clear the live bit of each
 * (request, token position) pair; the slot then reads as the sentinel dead
 * slot (logit -1e4, V = 0).  Token positions count appended tokens from 0.
 * req_ids: host int32 [n]; token_pos: host int64 [n].  Evicting twice is a no-op. */
KVQ_API kv_status_t kv_evict_slots(kv_pool_t* pool, const int32_t* req_ids, const int64_t* token_pos, int64_t n,
                           void* stream);

/* Per-head exclusion (HyQuant, core method: each key position belongs to
 * exactly one of the quantized set, the vertical-line set and the window of a
 * head, and vertical lines are chosen per kv head).  For each i, slot
 * token_pos[i] of request req_ids[i] reads as the sentinel dead slot for kv
 * head kv_heads[i] only; the other heads still read it.  The exclusion moves
 * with the slot when a staging page is requantized to INT2.
 * req_ids, kv_heads: host int32 [n]; token_pos: host int64 [n].  The first call
 * allocates one 32-bit word per (page, kv head) on the device and makes both
 * decode scans read it.  Excluding twice is a no-op; an invalid entry fails
 * the call before any change (KV_ERR_INVALID_ARG).
 * Per-head budgets (Tangram: head groups keep different amounts of context)
 * are this call applied to the positions outside a head's budget: the
 * tensor-core decode then skips every full page with no live slot for the
 * head, and the split plan balances the pages each head still reads. */
KVQ_API kv_status_t kv_evict_slots_head(kv_pool_t* pool, const int32_t* req_ids, const int64_t* token_pos,
                                        const int32_t* kv_heads, int64_t n, void* stream);

/* Free the pages nothing reads any more (Tangram: a head group holds only the
 * pages of its own budget; IntentKV method 2: surviving pages do not move).
 * For each listed request, every full page (32 tokens written) with no live
 * slot for any kv head (evicted, or excluded for every head) leaves the
 * table; the other entries keep their order, so positions and outputs are
 * unchanged (a dead slot adds exactly 0).  The freed ids return to their free
 * list and are reused lowest first.  Token positions of a dropped page stay
 * counted (kv_request_info) and read as gone: evicting or excluding them
 * again is a no-op.  req_ids: host int32 [n_req]; a request that is not open
 * fails the call before any change (KV_ERR_INVALID_ARG).  Partial pages (the
 * INT4 tail, the staging page) are kept. */
KVQ_API kv_status_t kv_drop_dead_pages(kv_pool_t* pool, const int32_t* req_ids, int32_t n_req, void* stream);

/* Full-precision token lists (HyQuant, Algorithm 3 and Algorithm 4 FREEZE:
 * the vertical-line tokens, the staging buffer and the window stay in full
 * precision and are scanned after the quantized prefix under the same online
 * softmax state).  Each request has one ordered list per kv head, every head
 * the same length and its own rows; kv_decode_attn scans the quantized pages,
 * then the list, and merges both with the split partials.  Which tokens a list
 * holds is the caller's choice (e.g. a head's vertical lines, excluded from
 * its quantized set with kv_evict_slots_head, and the most recent tokens).
 *
 * kv_fp_configure: capacity of every list in tokens (device memory:
 * 2 x max_requests x num_kv_heads x max_tokens x 256 bytes); 0 frees it.
 * Every list must be empty.  Synchronizes the device. */
KVQ_API kv_status_t kv_fp_configure(kv_pool_t* pool, int32_t max_tokens);

/* Append n_tok tokens to the lists: token t goes to the end of request
 * req_ids[t]'s lists, tokens of one request in order.
 *   k, v     device, bf16 [n_tok][num_kv_heads][128] (row h of token t goes to
 *            kv head h's list); any 2-byte alignment.
 *   req_ids  host, int32 [n_tok].
 * The values are used as given.  KV_ERR_OOM past a list's capacity and
 * KV_ERR_INVALID_ARG for a request that is not open, both before any change. */
KVQ_API kv_status_t kv_fp_append(kv_pool_t* pool, const void* k, const void* v, const int32_t* req_ids,
                                 int64_t n_tok, void* stream);

/* Remove list tokens [first, first + n_tok) of every head of a request; the
 * rest keep their order.  A range outside the list is KV_ERR_INVALID_ARG. */
KVQ_API kv_status_t kv_fp_drop(kv_pool_t* pool, int32_t req_id, int64_t first, int64_t n_tok, void* stream);

/* Host output: the length of a request's lists. */
KVQ_API kv_status_t kv_fp_count(kv_pool_t* pool, int32_t req_id, int64_t* n_tok);

/* Decode-step GQA attention over the page tables (TriAxialKV key design 4,
 * HyQuant Algorithm 3).
 *   q        device, bf16 [batch][num_q_heads][128]
 *   req_ids  host, int32 [batch]: request of each batch row
 *   out      device, fp32 [batch][num_q_heads][128]
 * q head h uses kv head h / (num_q_heads / num_kv_heads); num_q_heads must be
 * a multiple of num_kv_heads with a ratio <= 8.  A request with no tokens
 * yields zeros.  Logits are softmax_scale * q.k^ in fp32 accumulation. */
KVQ_API kv_status_t kv_decode_attn(kv_pool_t* pool, const void* q, const int32_t* req_ids, int32_t batch,
                           int32_t num_q_heads, float softmax_scale, float* out, void* stream);

/* Decode that allocates no device memory.  The pages have no counterpart for
 * this call; it exists for callers that cannot call cudaMalloc while they
 * decode: code whose device memory is owned entirely by another allocator or
 * a fixed budget (a framework's caching allocator, a serving loop that
 * reserved all memory up front), and latency-critical loops where a
 * cudaMalloc/cudaFree, which may synchronize the device, is not acceptable.
 * Same arguments, results and error rules as kv_decode_attn, except:
 *   - the split plan, the per-unit q operands and the split partials live in
 *     one fixed 64 MiB array inside the library (held on every GPU that loads
 *     it until the process exits) instead of pool buffers that grow with
 *     cudaMalloc; the call allocates nothing and frees nothing;
 *   - batch x num_kv_heads must be <= 4096 and the plan must fit the array
 *     (the worker count is lowered until it does); otherwise
 *     KV_ERR_INVALID_ARG with a message, before any device work;
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins;
 *   - each call copies its plan from pageable host memory with
 *     cudaMemcpyAsync on `stream`;
 *   - every call shares the array, which keeps the last call's contents;
 *     nothing in it has to start at zero (each call copies its plan in, and
 *     its scan writes every partial its merge reads); calls whose device work
 *     overlaps (other streams, other pools) race, so serialize them;
 *   - `stream` must be the stream that carries the pool's other work: this
 *     call neither waits for work the pool issued on another stream nor makes
 *     later pool calls wait for it, so on any other stream its ordering
 *     against appends, reorders and evictions is undefined;
 *   - kv_last_decode_stats and kv_decode_timing do not cover it.
 * The caller still provides q, out and the pool, as for kv_decode_attn. */
KVQ_API kv_status_t kv_decode_attn_noalloc(kv_pool_t* pool, const void* q, const int32_t* req_ids, int32_t batch,
                                           int32_t num_q_heads, float softmax_scale, float* out, void* stream);

/* Decode over head groups held in pools of their own (Tangram: head groups
 * keep different amounts of context).  Pool p holds kv heads
 * [h_p, h_p + num_kv_heads_p) of the model, h_p the kv heads of the pools
 * before it, fed the same tokens as the others but evicting (and dropping,
 * kv_drop_dead_pages) what its own budget leaves out, so it keeps only its
 * own pages.  One launch of the tensor-core scan walks every pool.
 *   pools    host [n_pools], 1 <= n_pools <= 8, distinct pools on one device
 *   q        device, bf16 [batch][num_q_heads][128]
 *   req_ids  host, int32 [n_pools][batch]: pool p's request of batch row b
 *   out      device, fp32 [batch][num_q_heads][128]
 * q head h uses kv head h / (num_q_heads / K) of the model, K the kv heads of
 * all pools together; num_q_heads must be a multiple of K with a ratio <= 8.
 * Results equal kv_decode_attn on one pool with all K heads in which each
 * head's excluded positions read as dead.  The scan skips every page with no
 * live slot for the head it reads it for.  Always the tensor-core scan,
 * whatever kv_set_decode_impl chose; pools may hold INT3 and FP4 pages.
 * Requests holding full-precision list tokens are KV_ERR_INVALID_ARG.  The plan, the q operands and the partials
 * live in pools[0]'s buffers, and a timeout of the scan is reported by
 * pools[0]'s kv_pool_sync; every pool's later work on another stream waits
 * for this call.  kv_last_decode_stats of each pool gives the bytes and
 * pages of its share (its split count is not updated); kv_decode_timing of
 * pools[0] covers the call. */
KVQ_API kv_status_t kv_decode_attn_groups(kv_pool_t* const* pools, int32_t n_pools, const void* q,
                                          const int32_t* req_ids, int32_t batch, int32_t num_q_heads,
                                          float softmax_scale, float* out, void* stream);

/* Testing aid for the device-timeout path (off by default).  Every copy wait
 * in the scans is bounded; first_wait_spins >= 0 makes the first copy wait of
 * every warp of the tensor-core page scan and of the full-precision list scan
 * give up after that many polls (0: at once) instead of the normal bound;
 * -1 restores the normal bound.  A warp whose wait gives up records
 * KV_ERR_DEVICE_TIMEOUT in the pool's status, still waits (with the normal
 * bound) for every copy it issued, writes empty partials and exits, so the
 * device stays usable: kv_pool_sync() then returns KV_ERR_DEVICE_TIMEOUT once
 * and the decode's output is unspecified.  Values outside [-1, 2^32) are
 * KV_ERR_INVALID_ARG. */
KVQ_API kv_status_t kv_set_wait_limit(kv_pool_t* pool, int64_t first_wait_spins);

/* Choose the decode implementation (kv_decode_impl_t). */
KVQ_API kv_status_t kv_set_decode_impl(kv_pool_t* pool, int32_t impl);

/* Wait for the pool's enqueued work; report device-side errors recorded since
 * the last call (KV_ERR_RANGE, KV_ERR_DEVICE_TIMEOUT) or KV_ERR_CUDA. */
KVQ_API kv_status_t kv_pool_sync(kv_pool_t* pool);

/* Host outputs: number of table entries and of appended tokens of a request. */
KVQ_API kv_status_t kv_request_info(kv_pool_t* pool, int32_t req_id, int32_t* n_pages, int64_t* n_tokens);

/* Canonical, synchronous export of one request, pages in table order (host
 * buffers sized from kv_request_info):
 *   ids [n], is_int2 [n], fill [n] (tokens written), live [n] (bit t = slot t live)
 *   k_codes, v_codes  uint8 [n][num_kv_heads][32][128]  (slot, channel)
 *   k_meta            uint16 [n][num_kv_heads][256]: INT4 / INT3 / FP4 page -> [slot][group]{scale, zero},
 *                     INT2 page -> [channel]{scale, zero}   (binary16 bits)
 *   v_meta            uint16 [n][num_kv_heads][256]: [slot][group]{scale, zero}
 * An INT3 page's codes are 0..7; an FP4 page's codes are E2M1 codes (sign <<
 * 3 | exponent << 1 | mantissa) with zero entries 0, its value = scale *
 * E2M1(code).  The width of a page follows from its id (n_int2_pages,
 * n_int4_pages, n_int3_pages ranges).  The four content pointers may all be
 * NULL to export the table only.  Slots at or past `fill` hold unspecified
 * content. */
KVQ_API kv_status_t kv_export_request(kv_pool_t* pool, int32_t req_id, int32_t* ids, uint8_t* is_int2, uint8_t* fill,
                              uint32_t* live, uint8_t* k_codes, uint8_t* v_codes, uint16_t* k_meta,
                              uint16_t* v_meta);

/* Algorithmic bytes and split count of the most recent kv_decode_attn call:
 * codes + scale/zero of every page block read (partial INT4, INT3 and FP4
 * pages count their filled prefix: 160, 128 and 144 bytes per token and kv
 * head), 8 bytes per table entry, q (bf16) and out (fp32), and the bf16 K and
 * V rows of the full-precision lists. */
KVQ_API kv_status_t kv_last_decode_stats(kv_pool_t* pool, int64_t* kv_bytes, int32_t* n_splits, int64_t* n_pages);

/* Device-time measurement of the decode kernels.  enable = N >= 1 starts (or
 * restarts) recording: every N-th later kv_decode_attn call (the first, the
 * (N+1)-th, ...) records CUDA events on its stream before the split scan,
 * between scan and merge, and after the merge (the last 2048 recorded calls
 * are kept).  The event between scan and merge keeps the merge from being
 * set up while the scan drains, so sampling (N > 1) leaves the other calls
 * undisturbed.  enable = 0 stops recording; enable < 0 is KV_ERR_INVALID_ARG.  On
 * return (host outputs, each may be NULL): *n_calls = calls recorded since the
 * last start (at most 2048 are averaged), *scan_ms / *decode_ms = mean duration
 * of the scan kernel / of scan + merge over them (waits for the last call's
 * events; -1 when no call was recorded). */
KVQ_API kv_status_t kv_decode_timing(kv_pool_t* pool, int32_t enable, int64_t* n_calls, float* scan_ms,
                                     float* decode_ms);

/* Number of kernels this pool has launched so far (host counter). */
KVQ_API kv_status_t kv_pool_launch_count(kv_pool_t* pool, int64_t* n_launches);

/* Greedy INT2/INT4 bit allocation (TriAxialKV key design 2), host only.
 * All tags start at 2 bits; tags with N_k > 0 are ranked by
 * rho_k = (D_k(2) - D_k(4)) / (2 N_k), descending (ties: lower tag first), and
 * raised to 4 bits whenever sum_k N_k b_k <= (B_num / B_den) sum_k N_k still
 * holds (a tag that does not fit is skipped).  N, D2, D4: host [n_tags];
 * bits_out: host uint8 [n_tags]. */
KVQ_API kv_status_t kv_alloc_bits(const int64_t* N, const double* D2, const double* D4, int32_t n_tags, int64_t B_num,
                          int64_t B_den, uint8_t* bits_out);

/* Greedy allocation over three widths (TriAxialKV, key design 2, with the
 * INT3 width its limitations and outlook section names): every tag starts at
 * 2 bits; its 2 -> 3 step saves D2[k] - D3[k], its 3 -> 4 step
 * D3[k] - D4[k], each costing N_k bit-tokens.  The available step with the
 * most distortion saved per bit-token goes first (a tag's 3 -> 4 step
 * becomes available once its 2 -> 3 step is taken; ties: the lower tag); a
 * step that does not fit sum_k N_k b_k <= (B_num / B_den) sum_k N_k (exact
 * integer test) is dropped and the scan continues.  With D3 = (D2 + D4) / 2
 * and room for whole upgrades only, the result is kv_alloc_bits's.
 *   N, D2, D3, D4  host [n_tags];  bits_out  host uint8 [n_tags] in {2, 3, 4}. */
KVQ_API kv_status_t kv_alloc_bits3(const int64_t* N, const double* D2, const double* D3, const double* D4,
                                   int32_t n_tags, int64_t B_num, int64_t B_den, uint8_t* bits_out);

/* Message for the calling thread's most recent failure ("" if none). */
KVQ_API const char* kv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
