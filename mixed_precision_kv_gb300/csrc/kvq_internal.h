// Internal state of a kv_pool_t and the launch interfaces shared by the
// library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <memory>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "../../include/kvq.h"
#include "kvq_layout.cuh"

namespace kvq {

// Device status word bits (OR-ed by kernels, read and cleared by kv_pool_sync).
constexpr uint32_t kStatusRange = 1u;
constexpr uint32_t kStatusTimeout = 2u;

// One table entry as the kernels read it.
struct Entry {
  int32_t id;
  uint32_t live;
};

// Host -> device table update, applied by a scatter kernel.
struct TableUpd {
  uint32_t index;   // kind 0: flat entry index r * max_pages + i; kind 1: request r; kind 2: page id
  int32_t a;        // kind 0: page id; kind 1: table length; kind 2: kv head
  uint32_t b;       // kind 0: live mask; kind 2: the page's slots excluded for that head
  uint32_t kind;
};

// Append job: one destination page and the tokens written into it this call.
struct AppendJob {
  int32_t page;        // INT4 page id (absolute; an INT3 id for the INT3 append kernel)
  int32_t first_slot;  // slot of the first token of this job (0: the page is new, its block starts from zeros)
  int32_t n_slots;     // tokens written by this job
  int32_t tok_off;     // offset into the token index list
  int32_t tab_index;   // flat index of the page's table entry after the call (-1: not in a table)
  uint32_t live;       // the page's live mask after the call
  int32_t ntab_req;    // request whose table length to set (-1: none)
  int32_t ntab_len;    // that length
};

// The jobs of a small append call, passed to the kernel by value (no copy).
struct SmallAppend {
  static constexpr int kMaxJobs = 32, kMaxToks = 128;
  AppendJob jobs[kMaxJobs];
  int32_t toks[kMaxToks];
};

struct RepackJob {
  int32_t src;  // INT4 staging page id
  int32_t dst;  // INT2 page id
};

// Direct INT2 job: 32 tokens of one request that fill a staging page within a
// single call, quantized to INT4, dequantized and requantized to INT2 in one
// kernel (the staging page is never written).
struct DirectJob {
  int32_t dst;      // INT2 page id
  int32_t tok_off;  // offset of its 32 token indices (slot order)
};

// Work unit of the decode: one (batch row, kv head).  Its splits (page ranges,
// one partial each) are contiguous in the split list, and so are the splits
// of its full-precision tokens (after every unit's page splits).
struct Unit {
  int32_t b;            // batch row
  int32_t req;          // request id
  int32_t kvh;          // kv head
  int32_t split_begin;  // first split of this unit
  int32_t n_splits;     // number of splits (0 = no tokens)
  int32_t fp_begin;     // first full-precision split of this unit
  int32_t n_fp_splits;  // number of full-precision splits
  int32_t pad;
};

// Full-precision splits: a Split whose page_begin / page_end are token
// indices of the request's lists (page_end < 0: to the list's length at
// launch).  The list tokens of all units, in unit order, are cut into ranges
// of about equal length, one per warp of the full-precision scan (at least
// kFpMinTokens tokens each), each range split further at unit boundaries.
constexpr int kFpWarpsPerCta = 8;
constexpr int kFpMinTokens = 32;

// A split: a range of one unit's pages in scan order, scanned by one worker
// (a CTA of the CUDA-core scan, a warp of the tensor-core scan).  Worker k
// scans the contiguous split range [cta_split[k], cta_split[k + 1]).
struct Split {
  int32_t unit;
  int32_t page_begin;   // scan-order position range [page_begin, page_end)
  int32_t page_end;     // < 0: to the end of the request's table (its device length at launch)
  int32_t req;          // request id of the unit
  int32_t n_pos;        // the unit's table length when planned
  int32_t n_lead;       // leading table entries spread evenly through the scan order (0: table order)
  int32_t pad[2];
};

// One pool of a grouped decode (kv_decode_attn_groups): its splits carry the
// pool's index (Split::pad[0]) and the kv head within the pool (pad[1]), its
// units the pool's index (Unit::pad), and the kernels read the pool's
// addresses from an array of these.
struct GroupPool {
  const uint8_t* pool;
  size_t int4_off;
  int64_t n2;
  const Entry* table;
  const int32_t* ntab;
  const uint32_t* hdead;   // null: no per-head exclusion in this pool
  const uint32_t* smax;    // the pool's largest INT2 K scale and largest V scale (float bits)
  size_t int3_off, fp4_off;  // INT3 / FP4 regions
  int64_t n3b, nfb;        // first INT3 and first FP4 id (no such pages: ids never reach them)
  int32_t hkv;
  int32_t max_pages;
  int32_t n_pools;         // entries in the array (the same in every entry)
  int32_t pad;
};
constexpr int kMaxGroupPools = 8;

// A full-precision scan to run between the page scan and the merge of the
// next decode launch (set by the caller of launch_decode_*).
struct FpLaunch {
  const Split* d_fsplits = nullptr;
  const int32_t* d_fpw = nullptr;
  int n_fpw = 0;
  int first_split = 0;
};

// Scan order of a unit: position p < n visits table index
//   lead  floor(p m / n)                 if floor((p+1) m / n) > floor(p m / n)
//   tail  m + p - floor((p+1) m / n)     otherwise,
// a bijection of [0, n) that spreads the m leading entries (the INT2 pages of
// a table sorted INT2-first) evenly among the others, so that every position
// range holds both precisions in the table's proportion; positions >= n
// (pages appended after planning) visit themselves.  Walked incrementally:
// a = floor(p m / n), rem = p m mod n.
struct ScanOrder {
  int32_t p, n, m, a, rem;
  __host__ __device__ void start(int32_t p0, int32_t n_, int32_t m_) {
    p = p0;
    n = n_;
    m = m_;
    const int64_t pm = (int64_t)p0 * m_;
    a = (n_ > 0 && p0 < n_) ? (int32_t)(pm / n_) : 0;
    rem = (n_ > 0 && p0 < n_) ? (int32_t)(pm % n_) : 0;
  }
  __host__ __device__ int32_t next() {   // table index of position p, then p + 1
    int32_t idx = p;
    if (p < n) {
      rem += m;
      if (rem >= n) {
        rem -= n;
        idx = a++;
      } else {
        idx = m + (p - a);
      }
    }
    ++p;
    return idx;
  }
};

// Planner cost of one page by precision, proportional to the scan kernel's
// time per page.  In the tensor-core scan an INT2 page costs more issue
// slots than an INT4 page: fitted to per-warp scan times of the 32K-token
// batch-8 (g = 4) and 100K-token batch-16 (g = 8) steps, an INT2 page takes
// 1.18x and 1.5x an INT4 page.  The CUDA-core scan is charged its block
// bytes plus 2048.
struct PageCost {
  double int2, int4, int3, fp4 = 1.0;
};
// INT3 pages: the INT4 page's work plus the assembly of every code from two
// planes; fitted the same way (32K-token batch-8 and 100K-token batch-16
// steps with every INT4 token made INT3): 1.28x and 1.40x an INT4 page.
// FP4 pages: a conversion per A register and no zero term, 1.06x an INT4
// page at g = 4 (the g = 8 figure assumed a little higher).
inline PageCost mma_page_cost(int g) {
  return g <= 4 ? PageCost{1.18, 1.00, 1.28, 1.06} : PageCost{1.50, 1.00, 1.40, 1.10};
}
constexpr PageCost kSimtPageCost{3072.0 + 2048.0, 5120.0 + 2048.0, 4096.0 + 2048.0, 4608.0 + 2048.0};
constexpr int64_t kMinPagesPerCta = 16;    // CUDA-core scan: pages per CTA at least
constexpr int64_t kMinPagesPerWarp = 1;    // tensor-core scan: pages per warp at least (small batches: more warps, less latency)
constexpr int64_t kTimingRing = 2048;

// Decode plan on the host (see plan_decode).
struct HostPlan {
  std::vector<Unit> units;
  std::vector<Split> splits;        // page splits, then full-precision splits
  int32_t n_page_splits = 0;
  std::vector<int32_t> fp_wsplit;   // full-precision workers + 1 entries (split indices from n_page_splits)
  std::vector<int32_t> cta_split;   // n_workers + 1 entries
  int64_t n_ctas() const { return (int64_t)cta_split.size() - 1; }   // workers
};

// Token positions of one request are int32 in the position maps: a request
// holds at most this many (appends past it are rejected before any change).
constexpr int64_t kMaxPositions = INT32_MAX;

// An allocator whose value-initialisation leaves a trivial element
// unwritten: resize() then grows a map without first storing zeros into
// entries that the caller writes right after.
template <class T>
struct NoFillAlloc : std::allocator<T> {
  template <class U>
  struct rebind {
    using other = NoFillAlloc<U>;
  };
  NoFillAlloc() = default;
  template <class U>
  NoFillAlloc(const NoFillAlloc<U>&) noexcept {}
  template <class U>
  void construct(U* p) noexcept {
    ::new ((void*)p) U;
  }
  template <class U, class... A>
  void construct(U* p, A&&... a) {
    ::new ((void*)p) U(std::forward<A>(a)...);
  }
};

struct Request {
  bool open = false;
  std::vector<int32_t> table;       // page ids in table order
  int32_t tail4 = -1, tail3 = -1, tailf = -1, staging = -1;
  std::vector<uint32_t, NoFillAlloc<uint32_t>> loc;   // token position -> page_id << 5 | slot
  uint64_t version = 0;             // bumped whenever the table's entries change
  uint64_t ordered_version = ~0ull; // version at which the table was last seen INT2-first
  uint64_t shape = 0;               // pool clock at the last open, erase or reorder of entries (not appends)
};

// Free page ids of one class, handed out lowest id first (a bitset with a
// hint at the lowest word that may hold a free id).
class FreeIds {
 public:
  void init(int32_t first, int32_t n) {
    first_ = first;
    bits_.assign((size_t)((n + 63) / 64), ~0ull);
    if (n % 64) bits_.back() = (1ull << (n % 64)) - 1;
    count_ = (size_t)n;
    lo_ = 0;
  }
  size_t size() const { return count_; }
  bool empty() const { return count_ == 0; }
  void insert(int32_t id) {
    const int32_t x = id - first_;
    uint64_t& wd = bits_[(size_t)(x >> 6)];
    const uint64_t b = 1ull << (x & 63);
    if (!(wd & b)) {
      wd |= b;
      ++count_;
      if ((size_t)(x >> 6) < lo_) lo_ = (size_t)(x >> 6);
    }
  }
  int32_t take_lowest() {   // caller ensures !empty()
    while (bits_[lo_] == 0) ++lo_;
    const int b = __builtin_ctzll(bits_[lo_]);
    bits_[lo_] &= bits_[lo_] - 1;
    --count_;
    return first_ + (int32_t)(lo_ * 64) + b;
  }

 private:
  std::vector<uint64_t> bits_;
  size_t count_ = 0, lo_ = 0;
  int32_t first_ = 0;
};

// A device buffer that grows geometrically (contents not preserved).
struct DevBuf {
  void* ptr = nullptr;
  size_t cap = 0;
};

}  // namespace kvq

struct kv_pool {
  kv_pool_config_t cfg;
  int sm_count = 0;
  // device memory
  uint8_t* d_pool = nullptr;          // INT2 region then INT4 region
  size_t pool_bytes = 0;
  size_t int4_offset = 0;             // byte offset of the INT4 region
  size_t int3_offset = 0;             // byte offset of the INT3 region (after the INT4 region)
  size_t fp4_offset = 0;              // byte offset of the FP4 region (after the INT3 region)
  kvq::Entry* d_table = nullptr;      // [max_requests][max_pages]
  int32_t* d_ntab = nullptr;          // [max_requests]
  uint32_t* d_status = nullptr;       // [0] status bits, [1] largest INT2 K scale, [2] largest V scale (fp32 bits)
  kvq::DevBuf upload;                 // append/scatter job arrays
  // pinned host staging of host-to-device copies (a ring: a slot is reused
  // once the copy recorded on its event has run)
  struct PinnedSlot {
    void* ptr = nullptr;
    size_t cap = 0;
    cudaEvent_t ev = nullptr;
    bool pending = false;
  };
  static constexpr int kPinnedSlots = 4;
  PinnedSlot pinned[kPinnedSlots];
  int pinned_next = 0;
  // host scratch reused by every call (kept at capacity: fresh vectors cost
  // an allocation and first-touch page faults per call)
  std::vector<int32_t> scr_i4, scr_i2, scr_toks, scr_dtoks;
  kvq::DevBuf plan;                   // decode plan (units, splits)
  kvq::DevBuf partials;               // decode split partials
  kvq::DevBuf frags;                  // per-unit q operands of the tensor-core scan
  // per-head exclusion (allocated by the first kv_evict_slots_head): per page
  // id x kv head, the slots that read as dead for that head only
  uint32_t* d_hdead = nullptr;
  std::vector<uint32_t> hdead;
  // full-precision token lists: K and V bf16 [max_requests][kv head][fp_cap][128]
  uint16_t* d_fpk = nullptr;
  uint16_t* d_fpv = nullptr;
  int32_t* d_nfp = nullptr;           // [max_requests] list lengths, written in stream order
  int32_t fp_cap = 0;
  std::vector<int32_t> n_fp;          // host mirror of the lengths
  kvq::DevBuf fp_scratch;             // kv_fp_drop staging
  // host mirror
  std::vector<kvq::Request> reqs;
  std::vector<uint8_t> fill;          // per page id
  std::vector<uint32_t> live;         // per page id
  std::vector<int32_t> pos;           // per page id x 32 slots: token position
  kvq::FreeIds free2, free3, free4, freef;
  std::vector<int32_t> call_slot;     // per request: index of its state inside the running append call (-1 outside)
  std::vector<int32_t> page_job;      // per page id: its append job inside the running call (-1 outside)
  // decode plan cache
  std::vector<int32_t> plan_req;
  std::vector<int32_t> plan_len;      // table lengths of plan_req when the plan was built
  std::vector<int32_t> plan_nfp;      // full-precision list lengths when the plan was built
  std::vector<uint64_t> plan_ver;     // table shapes (Request::shape) when the plan was built
  uint64_t shape_clock = 0;
  int32_t plan_slack = 0;             // pages a table may grow before the plan is rebuilt
  int32_t plan_hq = 0;
  int32_t plan_impl = -1;
  int32_t n_units = 0, n_splits = 0;
  int32_t n_page_splits = 0;          // splits [0, n_page_splits) are page splits, the rest full-precision
  size_t plan_fpw_off = 0;            // full-precision worker split ranges in the plan buffer
  kvq::FpLaunch fp_pending;           // launched by the next launch_decode_* between scan and merge
  int32_t n_fpw = 0;
  size_t plan_units_off = 0, plan_splits_off = 0, plan_cta_off = 0;
  int32_t n_ctas = 0;
  std::vector<int32_t> stat_req;      // request ids of the last decode (for kv_last_decode_stats)
  int32_t stat_hq = 0;
  bool stat_skip_dead = false;        // the last decode skipped pages with no live slot for a head
  // grouped decode plan cache (kv_decode_attn_groups with this pool first)
  uint64_t serial = 0;                        // unique per pool created in this process
  kvq::DevBuf gplan;
  std::vector<kvq::GroupPool> gplan_pools;    // the pools' descriptors when the plan was built
  std::vector<uint64_t> gplan_owner;          // and the pools' serials
  std::vector<int32_t> gplan_req, gplan_len;  // per (pool, batch row): request id and table length
  std::vector<uint64_t> gplan_ver;            // per (pool, batch row): table shape
  int32_t gplan_hq = 0, gplan_slack = 0;
  int32_t gplan_units = 0, gplan_splits = 0, gplan_workers = 0;
  size_t gplan_units_off = 0, gplan_splits_off = 0, gplan_wsplit_off = 0, gplan_pools_off = 0;
  int32_t decode_impl = KV_DECODE_AUTO;
  cudaStream_t last_stream = nullptr;
  int64_t launches = 0;               // kernels launched by this pool
  bool timing = false;                // record events around the decode kernels
  int32_t timing_every = 1;           // record every timing_every-th decode call
  int64_t timing_seen = 0;            // decode calls since timing started
  int64_t timed_calls = 0;            // decode calls recorded since timing started
  std::vector<cudaEvent_t> tev;       // ring of [before scan, after scan, after merge] per call
  cudaEvent_t merge_event = nullptr;  // recorded by the launchers between scan and merge when timing
  int64_t first_wait_spins = -1;      // kv_set_wait_limit: bound of the scans' first copy wait (-1: normal)
};

namespace kvq {

// Launch with programmatic stream serialization: the grid may be staged while
// the previous kernel of the stream drains.  Every kernel launched this way
// executes griddepcontrol.wait before it touches memory that earlier work in
// the stream reads or writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Sets the message kv_last_error() returns on this thread (kvq_pool.cu).
void set_last_error(const char* msg);

// Launchers (kvq_quant.cu)
cudaError_t launch_append(kv_pool* P, const void* k, const void* v, const AppendJob* d_jobs, int n_jobs,
                          const int32_t* d_toks, const SmallAppend* small, cudaStream_t s);
// INT3 tail pages (jobs whose page is an INT3 id)
cudaError_t launch_append_int3(kv_pool* P, const void* k, const void* v, const AppendJob* d_jobs, int n_jobs,
                               const int32_t* d_toks, cudaStream_t s);
// FP4 tail pages (jobs whose page is an FP4 id)
cudaError_t launch_append_fp4(kv_pool* P, const void* k, const void* v, const AppendJob* d_jobs, int n_jobs,
                              const int32_t* d_toks, cudaStream_t s);
cudaError_t launch_repack(kv_pool* P, const RepackJob* d_jobs, int n_jobs, cudaStream_t s);
cudaError_t launch_direct_int2(kv_pool* P, const void* k, const void* v, const DirectJob* d_jobs, int n_jobs,
                               const int32_t* d_toks, cudaStream_t s);
cudaError_t launch_scatter(kv_pool* P, const TableUpd* d_upd, int n, cudaStream_t s);
// Bulk forms (a warp per 32-channel group, a lane per token; K/V rows 16-byte
// aligned): fresh INT4 pages of 32 tokens, and direct INT2 groups.
cudaError_t launch_bulk_int4(kv_pool* P, const void* k, const void* v, const AppendJob* d_jobs, int n_jobs,
                             const int32_t* d_toks, cudaStream_t s);
cudaError_t launch_bulk_int2(kv_pool* P, const void* k, const void* v, const DirectJob* d_jobs, int n_jobs,
                             const int32_t* d_toks, cudaStream_t s);

// Balanced decode plan: units (batch row, kv head) in order, their pages cut
// into n_workers contiguous ranges of about equal cost (at least min_pages
// pages each), each range split further at unit boundaries (kvq_pool.cu).
// spread: splits walk each unit in its ScanOrder (INT2 pages interleaved);
// otherwise in table order.
void plan_decode(const kv_pool* P, const int32_t* req_ids, int32_t batch, int64_t n_workers, int64_t min_pages,
                 PageCost cost, bool spread, HostPlan& out);
int fp_workers(const kv_pool* P);   // warps of the full-precision scan (one CTA per SM)

// Full-precision scan (kvq_fp.cu): warp k scans the splits
// [d_fpw[k], d_fpw[k + 1]) of d_fsplits and writes one partial per split at
// split index first_split + i of d_part.  Launched as a programmatic
// dependent of the page scan (it reads nothing the scan writes and waits for
// the scan grid before it exits).  launch_fp_pending launches P->fp_pending
// and clears it.
cudaError_t launch_fp_segments(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units,
                               const Split* d_fsplits, const int32_t* d_fpw, int n_fpw, int first_split, float* d_part,
                               cudaStream_t s);
cudaError_t launch_fp_pending(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units,
                              float* d_part, cudaStream_t s);
// Copies into / within the full-precision lists (kvq_fp.cu).
cudaError_t launch_fp_store(kv_pool* P, const void* k, const void* v, int64_t n, const int32_t* d_req,
                            const int32_t* d_slot, const int32_t* d_len_req, const int32_t* d_len_val, int n_len,
                            cudaStream_t s);
cudaError_t launch_fp_move(kv_pool* P, int32_t req, int32_t from, int32_t to, int32_t n, int32_t new_len,
                           cudaStream_t s);

// Launchers (kvq_decode_simt.cu / kvq_decode_mma.cu)
cudaError_t launch_decode_simt(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units,
                               int n_units, const Split* d_splits, const int32_t* d_cta, int n_ctas, float* d_part,
                               float* out, cudaStream_t s);
int decode_simt_ctas_per_sm(int g);
// Tensor-core scan: workers are warps; d_frags holds decode_mma_frag_bytes()
// per unit (the q operands its per-unit kernel builds before the scan).
// Grouped form: d_gpools != null (device array of GroupPool) makes every
// unit and split name its pool; total_kv_heads is then the kv heads of all
// pools together (hq / total_kv_heads q heads per kv head); groups_extra:
// some pool holds INT3 or FP4 pages.
cudaError_t launch_decode_mma(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units, int n_units,
                              const Split* d_splits, const int32_t* d_wsplit, int n_workers, void* d_frags,
                              float* d_part, float* out, cudaStream_t s, const GroupPool* d_gpools = nullptr,
                              int32_t total_kv_heads = 0, bool groups_extra = false);
int decode_mma_workers_per_sm(int g);
constexpr int kMmaWarpsPerCta = 16;
size_t decode_mma_frag_bytes();
// Split merge: out[b][h][:] = sum_s acc_s 2^(m_s - M) / sum_s l_s 2^(m_s - M) over the unit's splits.
cudaError_t launch_merge(kv_pool* P, int g, const Unit* d_units, int n_units, const float* d_part, int hq, float* out,
                         cudaStream_t s);

}  // namespace kvq
