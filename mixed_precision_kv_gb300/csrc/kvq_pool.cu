// Host side of the C ABI: pool and request management, deterministic page
// allocation, token routing (INT4 tail / INT4 staging -> INT2 repack), INT2-
// first reorder, eviction, export, the decode split planner and the decode
// dispatch.  Every device step runs in the kernels of kvq_quant.cu and
// kvq_decode_*.cu; this file only decides what they do.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

#include "kvq_internal.h"

using namespace kvq;

namespace {

thread_local std::string g_err;

kv_status_t fail(kv_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

#define KV_CUDA(call)                                                                       \
  do {                                                                                      \
    cudaError_t e_ = (call);                                                                \
    if (e_ != cudaSuccess) return fail(KV_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

// Makes the pool's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool req_ok(const kv_pool* P, int32_t r) {
  return r >= 0 && r < P->cfg.max_requests && P->reqs[r].open;
}

bool is_int2(const kv_pool* P, int32_t id) { return id < P->cfg.n_int2_pages; }
// INT3 ids follow the INT2 and INT4 ids, FP4 ids the INT3 ids
int64_t first_int3(const kv_pool* P) { return P->cfg.n_int2_pages + P->cfg.n_int4_pages; }
int64_t first_fp4(const kv_pool* P) { return first_int3(P) + P->cfg.n_int3_pages; }
bool is_fp4(const kv_pool* P, int32_t id) { return id >= first_fp4(P); }
bool is_int3(const kv_pool* P, int32_t id) { return id >= first_int3(P) && id < first_fp4(P); }
// sort key of the reorder: INT2, INT3, INT4, FP4
int width_of(const kv_pool* P, int32_t id) { return is_int2(P, id) ? 2 : (is_int3(P, id) ? 3 : (is_fp4(P, id) ? 5 : 4)); }
FreeIds& free_list(kv_pool* P, int32_t id) {
  return is_int2(P, id) ? P->free2 : (is_int3(P, id) ? P->free3 : (is_fp4(P, id) ? P->freef : P->free4));
}

// Position-map entry of a token whose page was dropped (kv_drop_dead_pages).
constexpr uint32_t kDroppedLoc = 0xFFFFFFFFu;

// Per-head exclusion words (kept once kv_evict_slots_head has been used):
// host mirror changes, each queued as a kind-2 table update for the device.
void hdead_set(kv_pool* P, int32_t id, int h, uint32_t val, std::vector<TableUpd>& hu) {
  uint32_t& w = P->hdead[(size_t)id * P->cfg.num_kv_heads + h];
  if (w != val) {
    w = val;
    hu.push_back(TableUpd{(uint32_t)id, h, val, 2u});
  }
}
void hdead_copy(kv_pool* P, int32_t dst, int32_t src, std::vector<TableUpd>& hu) {
  if (P->hdead.empty()) return;
  for (int h = 0; h < P->cfg.num_kv_heads; ++h)
    hdead_set(P, dst, h, P->hdead[(size_t)src * P->cfg.num_kv_heads + h], hu);
}
void hdead_clear(kv_pool* P, int32_t id, std::vector<TableUpd>& hu) {
  if (P->hdead.empty()) return;
  for (int h = 0; h < P->cfg.num_kv_heads; ++h) hdead_set(P, id, h, 0u, hu);
}
// One update per word, carrying its final value: the scatter kernel applies
// updates in no particular order.
void hdead_final(const kv_pool* P, std::vector<TableUpd>& hu) {
  std::sort(hu.begin(), hu.end(), [](const TableUpd& x, const TableUpd& y) {
    return x.index != y.index ? x.index < y.index : x.a < y.a;
  });
  hu.erase(std::unique(hu.begin(), hu.end(),
                       [](const TableUpd& x, const TableUpd& y) { return x.index == y.index && x.a == y.a; }),
           hu.end());
  for (auto& u : hu) u.b = P->hdead[(size_t)u.index * P->cfg.num_kv_heads + u.a];
}


// Grow a device buffer to at least `bytes` (contents are not kept).
kv_status_t ensure(DevBuf& b, size_t bytes) {
  if (b.cap >= bytes) return KV_OK;
  size_t cap = std::max<size_t>(bytes, b.cap * 2);
  cap = (cap + 255) & ~size_t(255);
  if (b.ptr) {
    KV_CUDA(cudaDeviceSynchronize());
    KV_CUDA(cudaFree(b.ptr));
    b.ptr = nullptr;
    b.cap = 0;
  }
  KV_CUDA(cudaMalloc(&b.ptr, cap));
  b.cap = cap;
  return KV_OK;
}

// Several host arrays laid out for one upload (one H2D copy per call); the
// arrays are copied straight into the pinned staging buffer by h2d (they must
// stay alive until then).
struct Upload {
  struct Piece {
    const void* p;
    size_t n, off;
  };
  static constexpr int kMaxPieces = 8;
  Piece pieces[kMaxPieces];
  int n_pieces = 0;
  size_t size = 0;
  size_t add(const void* p, size_t n) {   // byte offset of the array in the upload
    const size_t off = (size + 255) & ~size_t(255);
    pieces[n_pieces++] = Piece{p, n, off};
    size = off + n;
    return off;
  }
};

// Host-to-device copy through a pinned staging slot.  A copy from pageable
// memory first waits for the stream to drain, which would stall the queue of
// calls the host keeps ahead of the GPU; from pinned memory it is queued like
// a kernel.  A slot is reused after its previous copy has run (normally long
// before: the ring has kPinnedSlots slots).
kv_status_t h2d(kv_pool* P, void* dst, const Upload& u, cudaStream_t s) {
  const size_t n = u.size;
  if (n == 0) return KV_OK;
  kv_pool::PinnedSlot& sl = P->pinned[P->pinned_next];
  P->pinned_next = (P->pinned_next + 1) % kv_pool::kPinnedSlots;
  if (sl.pending) {
    KV_CUDA(cudaEventSynchronize(sl.ev));
    sl.pending = false;
  }
  if (sl.cap < n) {
    if (sl.ptr) KV_CUDA(cudaFreeHost(sl.ptr));
    sl.ptr = nullptr;
    sl.cap = 0;
    const size_t cap = std::max(n + n / 2, size_t(1) << 16);
    KV_CUDA(cudaMallocHost(&sl.ptr, cap));
    sl.cap = cap;
  }
  if (!sl.ev) KV_CUDA(cudaEventCreateWithFlags(&sl.ev, cudaEventDisableTiming));
  for (int i = 0; i < u.n_pieces; ++i)
    if (u.pieces[i].n) std::memcpy((uint8_t*)sl.ptr + u.pieces[i].off, u.pieces[i].p, u.pieces[i].n);
  KV_CUDA(cudaMemcpyAsync(dst, sl.ptr, n, cudaMemcpyHostToDevice, s));
  KV_CUDA(cudaEventRecord(sl.ev, s));
  sl.pending = true;
  return KV_OK;
}

kv_status_t upload(kv_pool* P, const Upload& u, cudaStream_t s) {
  if (u.size == 0) return KV_OK;
  kv_status_t st = ensure(P->upload, u.size);
  if (st != KV_OK) return st;
  return h2d(P, P->upload.ptr, u, s);
}

// Device table rows to rewrite after a call: per request, every entry from
// `from` to the end plus individually listed entries below it.
struct Dirty {
  std::unordered_map<int32_t, int32_t> from;                // request -> first index to rewrite
  std::unordered_map<int32_t, std::vector<int32_t>> pages;  // request -> page ids whose live mask changed
  void structural(int32_t r, int32_t idx) {
    auto it = from.find(r);
    if (it == from.end()) from[r] = idx; else it->second = std::min(it->second, idx);
  }
  void live(int32_t r, int32_t page) { pages[r].push_back(page); }
};

void emit_updates(const kv_pool* P, const Dirty& d, std::vector<TableUpd>& out) {
  const uint32_t mp = (uint32_t)P->cfg.max_pages_per_request;
  std::unordered_map<int32_t, int32_t> f(d.from.begin(), d.from.end());
  for (const auto& kv : f) {
    const auto& tb = P->reqs[kv.first].table;
    for (int32_t i = kv.second; i < (int32_t)tb.size(); ++i)
      out.push_back(TableUpd{(uint32_t)kv.first * mp + (uint32_t)i, tb[i], P->live[tb[i]], 0u});
    out.push_back(TableUpd{(uint32_t)kv.first, (int32_t)tb.size(), 0u, 1u});
  }
  for (const auto& kv : d.pages) {
    const auto& tb = P->reqs[kv.first].table;
    const auto it = f.find(kv.first);
    const int32_t lim = it == f.end() ? INT_MAX : it->second;
    std::vector<int32_t> ids = kv.second;
    std::sort(ids.begin(), ids.end());
    ids.erase(std::unique(ids.begin(), ids.end()), ids.end());
    for (int32_t i = 0; i < (int32_t)tb.size() && i < lim; ++i)
      if (std::binary_search(ids.begin(), ids.end(), tb[i]))
        out.push_back(TableUpd{(uint32_t)kv.first * mp + (uint32_t)i, tb[i], P->live[tb[i]], 0u});
  }
}

// Order this call after the pool's previous work when the stream changes.
kv_status_t order_after_previous(kv_pool* P, cudaStream_t s) {
  if (P->last_stream != s && P->last_stream != nullptr) {
    cudaEvent_t ev;
    KV_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    KV_CUDA(cudaEventRecord(ev, P->last_stream));
    KV_CUDA(cudaStreamWaitEvent(s, ev, 0));
    KV_CUDA(cudaEventDestroy(ev));
  }
  P->last_stream = s;
  return KV_OK;
}

}  // namespace

void kvq::set_last_error(const char* msg) { g_err = msg; }

void kvq::plan_decode(const kv_pool* P, const int32_t* req_ids, int32_t batch, int64_t n_ctas, int64_t min_pages,
                       PageCost pc, bool spread, HostPlan& out) {
  const int hkv = P->cfg.num_kv_heads;
  const int64_t n2 = P->cfg.n_int2_pages, n3b = n2 + P->cfg.n_int4_pages, nfb = n3b + P->cfg.n_int3_pages;
  auto cost = [&](int32_t id) { return id < n2 ? pc.int2 : (id >= nfb ? pc.fp4 : (id >= n3b ? pc.int3 : pc.int4)); };
  // Per request: the cost of its first i pages in scan order (shared by the
  // request's kv heads), so that worker boundaries are found by binary search
  // instead of a walk over every (page, kv head).  With per-head exclusion
  // the prefix is per unit: a full page with no live slot for the head costs
  // nothing (the tensor-core scan skips it; a page still being filled keeps
  // its cost, since appends may give it live slots).
  const bool per_head = !P->hdead.empty();
  const int np = per_head ? hkv : 1;   // prefixes per request
  std::vector<int64_t> off((size_t)batch * np + 1, 0);
  std::vector<int32_t> lead((size_t)batch, 0);
  for (int32_t b = 0; b < batch; ++b) {
    const auto& tb = P->reqs[req_ids[b]].table;
    if (spread)
      for (int32_t id : tb) lead[b] += id < n2 ? 1 : 0;
    for (int x = 0; x < np; ++x) off[(size_t)b * np + x + 1] = off[(size_t)b * np + x] + (int64_t)tb.size() + 1;
  }
  std::vector<double> pre((size_t)off[(size_t)batch * np]);
  double total = 0.0;
  int64_t pages = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const auto& tb = P->reqs[req_ids[b]].table;
    const int32_t npos = (int32_t)tb.size();
    ScanOrder so;
    so.start(0, npos, lead[b]);
    for (int x = 0; x < np; ++x) pre[off[(size_t)b * np + x]] = 0.0;
    for (int32_t i = 0; i < npos; ++i) {
      const int32_t id = tb[so.next()];
      const double c = cost(id);
      for (int x = 0; x < np; ++x) {
        double* pb = &pre[off[(size_t)b * np + x]];
        const bool dead = per_head && P->fill[id] == kPage && (P->live[id] & ~P->hdead[(size_t)id * hkv + x]) == 0u;
        pb[i + 1] = pb[i] + (dead ? 0.0 : c);
      }
    }
    for (int x = 0; x < np; ++x) total += pre[off[(size_t)b * np + x] + npos] * (per_head ? 1 : hkv);
    pages += (int64_t)npos * hkv;
  }
  // at least min_pages pages per worker, so small batches do not pay a
  // worker's fixed cost per page
  const int64_t n = std::max<int64_t>(1, std::min<int64_t>(n_ctas, pages / std::max<int64_t>(1, min_pages)));
  out.units.assign((size_t)batch * hkv, Unit{});
  out.splits.clear();
  out.cta_split.assign((size_t)n + 1, 0);
  // page at cost offset c (cost of everything before it) goes to worker floor(c n / total)
  const double scale = total > 0.0 ? (double)n / total : 0.0;
  auto worker = [&](double c) { return std::min<int64_t>(n - 1, (int64_t)(c * scale)); };
  int64_t cur = 0;        // worker receiving the current split
  double U = 0.0;         // cost before the current unit
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t npos = (int32_t)P->reqs[req_ids[b]].table.size();
    for (int h = 0; h < hkv; ++h) {
      const double* pb = &pre[off[(size_t)b * np + (per_head ? h : 0)]];
      const int32_t ui = b * hkv + h;
      Unit& u = out.units[ui];
      u.b = b;
      u.req = req_ids[b];
      u.kvh = h;
      u.split_begin = (int32_t)out.splits.size();
      int32_t i = 0;
      if (per_head) {
        // leading full pages with no live slot for this head (a head that keeps
        // only recent tokens) are left out of the splits: no worker walks them.
        // The plan is rebuilt whenever a table's entries are erased or moved,
        // so the pages at those positions stay the ones found dead here (new
        // pages go to the end; exclusions and evictions only kill slots).
        while (i < npos && pb[i + 1] == pb[i]) ++i;
        if (i == npos && npos > 0) {
          // nothing live: one empty split, open-ended so that pages appended
          // after planning are scanned
          const int64_t j = worker(U + pb[npos]);
          while (cur < j) out.cta_split[++cur] = (int32_t)out.splits.size();
          out.splits.push_back(Split{ui, npos, npos, req_ids[b], npos, lead[b], {0, 0}});
        }
      }
      while (i < npos) {
        const int64_t j = worker(U + pb[i]);
        while (cur < j) out.cta_split[++cur] = (int32_t)out.splits.size();
        // first position after i that belongs to a later worker (npos: none)
        int32_t lo = i + 1, hi = npos;
        while (lo < hi) {
          const int32_t mid = lo + (hi - lo) / 2;
          if (worker(U + pb[mid]) > j) hi = mid;
          else lo = mid + 1;
        }
        out.splits.push_back(Split{ui, i, lo, req_ids[b], npos, lead[b], {0, 0}});
        i = lo;
      }
      U += pb[npos];
      u.n_splits = (int32_t)out.splits.size() - u.split_begin;
      // the unit's last split runs to the end of the table, so pages appended
      // after planning are scanned too (by the worker that owns the tail)
      if (u.n_splits > 0) out.splits.back().page_end = -1;
    }
  }
  while (cur < n) out.cta_split[++cur] = (int32_t)out.splits.size();
  // full-precision splits, after all page splits: the list tokens of all
  // units, in unit order, cut into fp_workers(P) ranges of about equal
  // length (at least kFpMinTokens each), split at unit boundaries; a unit's
  // last split runs to the list's length at launch
  out.n_page_splits = (int32_t)out.splits.size();
  int64_t T = 0;
  for (int32_t b = 0; b < batch; ++b) T += (int64_t)hkv * (P->n_fp.empty() ? 0 : P->n_fp[req_ids[b]]);
  const int64_t nw = T > 0 ? std::max<int64_t>(1, std::min<int64_t>(fp_workers(P), (T + kFpMinTokens - 1) / kFpMinTokens))
                           : 0;
  out.fp_wsplit.assign((size_t)nw + 1, 0);
  int64_t fcur = 0, FU = 0;   // worker receiving the current split; tokens before the current unit
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t nf = P->n_fp.empty() ? 0 : P->n_fp[req_ids[b]];
    for (int h = 0; h < hkv; ++h) {
      Unit& u = out.units[(size_t)b * hkv + h];
      u.fp_begin = (int32_t)out.splits.size();
      for (int32_t t = 0; t < nf;) {
        const int64_t j = (FU + t) * nw / T;   // worker of token t
        while (fcur < j) out.fp_wsplit[(size_t)++fcur] = (int32_t)out.splits.size() - out.n_page_splits;
        // first token of worker j + 1: ceil((j + 1) T / nw)
        const int64_t lim = ((j + 1) * T + nw - 1) / nw - FU;
        const int32_t e = (int32_t)std::min<int64_t>(nf, lim);
        out.splits.push_back(Split{b * hkv + h, t, e, req_ids[b], 0, 0, {0, 0}});
        t = e;
      }
      FU += nf;
      u.n_fp_splits = (int32_t)out.splits.size() - u.fp_begin;
      if (u.n_fp_splits > 0) out.splits.back().page_end = -1;
    }
  }
  while (fcur < nw) out.fp_wsplit[(size_t)++fcur] = (int32_t)out.splits.size() - out.n_page_splits;
}

extern "C" {

const char* kv_last_error(void) { return g_err.c_str(); }

kv_status_t kv_alloc_bits(const int64_t* N, const double* D2, const double* D4, int32_t n_tags, int64_t B_num,
                          int64_t B_den, uint8_t* bits_out) {
  if (!N || !D2 || !D4 || !bits_out || n_tags <= 0) return fail(KV_ERR_INVALID_ARG, "kv_alloc_bits: bad pointer or n_tags");
  if (B_den <= 0 || B_num < 0) return fail(KV_ERR_INVALID_ARG, "kv_alloc_bits: budget must be num >= 0, den > 0");
  int64_t total = 0;
  for (int32_t k = 0; k < n_tags; ++k) {
    if (N[k] < 0) return fail(KV_ERR_INVALID_ARG, "kv_alloc_bits: negative count");
    total += N[k];
  }
  // Rank tags by marginal distortion saved per extra bit-token.
  std::vector<int32_t> idx;
  std::vector<double> rho(n_tags, 0.0);
  for (int32_t k = 0; k < n_tags; ++k) {
    bits_out[k] = 2;
    if (N[k] > 0) {
      rho[k] = (D2[k] - D4[k]) / (2.0 * (double)N[k]);
      idx.push_back(k);
    }
  }
  std::sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) {
    return rho[a] != rho[b] ? rho[a] > rho[b] : a < b;
  });
  // Integer budget test: (used + 2 N_k) * den <= num * total.
  int64_t used = 2 * total;
  for (int32_t k : idx) {
    if ((used + 2 * N[k]) * B_den <= B_num * total) {
      bits_out[k] = 4;
      used += 2 * N[k];
    }
  }
  return KV_OK;
}

kv_status_t kv_alloc_bits3(const int64_t* N, const double* D2, const double* D3, const double* D4, int32_t n_tags,
                           int64_t B_num, int64_t B_den, uint8_t* bits_out) {
  if (!N || !D2 || !D3 || !D4 || !bits_out || n_tags <= 0)
    return fail(KV_ERR_INVALID_ARG, "kv_alloc_bits3: bad pointer or n_tags");
  if (B_den <= 0 || B_num < 0) return fail(KV_ERR_INVALID_ARG, "kv_alloc_bits3: budget must be num >= 0, den > 0");
  int64_t total = 0;
  for (int32_t k = 0; k < n_tags; ++k) {
    if (N[k] < 0) return fail(KV_ERR_INVALID_ARG, "kv_alloc_bits3: negative count");
    total += N[k];
    bits_out[k] = 2;
  }
  // One-bit steps in a max-heap keyed by distortion saved per bit-token
  // (ties: lower tag first); a tag's 3 -> 4 step enters once its 2 -> 3 step
  // is taken.  Integer budget test: (used + N_k) * den <= num * total.
  struct Step {
    double rho;
    int32_t tag;
  };
  auto later = [](const Step& a, const Step& b) { return a.rho != b.rho ? a.rho < b.rho : a.tag > b.tag; };
  std::vector<Step> heap;
  heap.reserve((size_t)n_tags);
  for (int32_t k = 0; k < n_tags; ++k)
    if (N[k] > 0) heap.push_back(Step{(D2[k] - D3[k]) / (double)N[k], k});
  std::make_heap(heap.begin(), heap.end(), later);
  int64_t used = 2 * total;
  while (!heap.empty()) {
    std::pop_heap(heap.begin(), heap.end(), later);
    const Step st = heap.back();
    heap.pop_back();
    const int32_t k = st.tag;
    if ((used + N[k]) * B_den > B_num * total) continue;   // dropped, with any later step of the tag
    used += N[k];
    if (bits_out[k] == 2) {
      bits_out[k] = 3;
      heap.push_back(Step{(D3[k] - D4[k]) / (double)N[k], k});
      std::push_heap(heap.begin(), heap.end(), later);
    } else {
      bits_out[k] = 4;
    }
  }
  return KV_OK;
}

kv_status_t kv_pool_create(const kv_pool_config_t* cfg, kv_pool_t** out) {
  if (!cfg || !out) return fail(KV_ERR_INVALID_ARG, "kv_pool_create: null argument");
  *out = nullptr;
  if (cfg->head_dim != kHeadDim || cfg->page_tokens != kPage || cfg->group != kGroup)
    return fail(KV_ERR_INVALID_ARG, "kv_pool_create: head_dim, page_tokens and group must be 128, 32, 32");
  if (cfg->num_kv_heads < 1 || cfg->num_kv_heads > 64)
    return fail(KV_ERR_INVALID_ARG, "kv_pool_create: num_kv_heads must be in [1, 64]");
  if (cfg->n_int2_pages < 0 || cfg->n_int4_pages < 1 || cfg->n_int3_pages < 0 || cfg->n_fp4_pages < 0 ||
      cfg->n_int2_pages + cfg->n_int4_pages + cfg->n_int3_pages + cfg->n_fp4_pages > (int64_t(1) << 27))
    return fail(KV_ERR_INVALID_ARG, "kv_pool_create: need n_int4_pages >= 1, n_int3_pages, n_fp4_pages >= 0 and "
                                    "at most 2^27 pages in total");
  if (cfg->max_requests < 1 || cfg->max_pages_per_request < 1 ||
      (int64_t)cfg->max_requests * cfg->max_pages_per_request > (int64_t(1) << 32) - 1)
    return fail(KV_ERR_INVALID_ARG, "kv_pool_create: bad max_requests / max_pages_per_request");
  int ndev = 0;
  KV_CUDA(cudaGetDeviceCount(&ndev));
  if (cfg->device < 0 || cfg->device >= ndev) return fail(KV_ERR_INVALID_ARG, "kv_pool_create: bad device %d", cfg->device);
  DeviceGuard dg(cfg->device);
  if (!dg.ok) return fail(KV_ERR_CUDA, "kv_pool_create: cudaSetDevice failed");

  kv_pool* P = new (std::nothrow) kv_pool();
  if (!P) return fail(KV_ERR_OOM, "kv_pool_create: host allocation failed");
  P->cfg = *cfg;
  static std::atomic<uint64_t> serials{0};
  P->serial = ++serials;
  auto cleanup = [&](kv_status_t st) {
    cudaFree(P->d_pool);
    cudaFree(P->d_table);
    cudaFree(P->d_ntab);
    cudaFree(P->d_status);
    delete P;
    return st;
  };
  if (cudaDeviceGetAttribute(&P->sm_count, cudaDevAttrMultiProcessorCount, cfg->device) != cudaSuccess)
    return cleanup(fail(KV_ERR_CUDA, "kv_pool_create: cannot query SM count"));
  const size_t hkv = (size_t)cfg->num_kv_heads;
  P->int4_offset = (size_t)cfg->n_int2_pages * hkv * kInt2Block;
  P->int3_offset = P->int4_offset + (size_t)cfg->n_int4_pages * hkv * kInt4Block;
  P->fp4_offset = P->int3_offset + (size_t)cfg->n_int3_pages * hkv * kInt3Block;
  P->pool_bytes = P->fp4_offset + (size_t)cfg->n_fp4_pages * hkv * kFp4Block;
  if (cudaMalloc(&P->d_pool, P->pool_bytes) != cudaSuccess) {
    cudaGetLastError();
    return cleanup(fail(KV_ERR_OOM, "kv_pool_create: cannot allocate %zu bytes of pool", P->pool_bytes));
  }
  const size_t tab = (size_t)cfg->max_requests * cfg->max_pages_per_request * sizeof(Entry);
  if (cudaMalloc(&P->d_table, tab) != cudaSuccess || cudaMalloc(&P->d_ntab, cfg->max_requests * 4) != cudaSuccess ||
      cudaMalloc(&P->d_status, 16) != cudaSuccess) {
    cudaGetLastError();
    return cleanup(fail(KV_ERR_OOM, "kv_pool_create: cannot allocate tables"));
  }
  if (cudaMemset(P->d_table, 0xFF, tab) != cudaSuccess || cudaMemset(P->d_ntab, 0, cfg->max_requests * 4) != cudaSuccess ||
      cudaMemset(P->d_status, 0, 16) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return cleanup(fail(KV_ERR_CUDA, "kv_pool_create: initialisation failed"));
  const size_t npages = (size_t)(cfg->n_int2_pages + cfg->n_int4_pages + cfg->n_int3_pages + cfg->n_fp4_pages);
  try {
    P->reqs.resize(cfg->max_requests);
    P->fill.assign(npages, 0);
    P->live.assign(npages, 0);
    P->pos.assign(npages * kPage, -1);
    P->free2.init(0, (int32_t)cfg->n_int2_pages);
    P->free4.init((int32_t)cfg->n_int2_pages, (int32_t)cfg->n_int4_pages);
    P->free3.init((int32_t)(cfg->n_int2_pages + cfg->n_int4_pages), (int32_t)cfg->n_int3_pages);
    P->freef.init((int32_t)(cfg->n_int2_pages + cfg->n_int4_pages + cfg->n_int3_pages), (int32_t)cfg->n_fp4_pages);
  } catch (...) {
    return cleanup(fail(KV_ERR_OOM, "kv_pool_create: host allocation failed"));
  }
  *out = P;
  return KV_OK;
}

kv_status_t kv_pool_destroy(kv_pool_t* P) {
  if (!P) return fail(KV_ERR_INVALID_ARG, "kv_pool_destroy: null pool");
  DeviceGuard dg(P->cfg.device);
  cudaDeviceSynchronize();
  cudaFree(P->d_pool);
  cudaFree(P->d_table);
  cudaFree(P->d_ntab);
  cudaFree(P->d_status);
  cudaFree(P->upload.ptr);
  cudaFree(P->plan.ptr);
  cudaFree(P->partials.ptr);
  cudaFree(P->frags.ptr);
  cudaFree(P->gplan.ptr);
  cudaFree(P->d_hdead);
  cudaFree(P->d_fpk);
  cudaFree(P->d_fpv);
  cudaFree(P->d_nfp);
  cudaFree(P->fp_scratch.ptr);
  for (cudaEvent_t e : P->tev)
    if (e) cudaEventDestroy(e);
  for (auto& sl : P->pinned) {
    if (sl.ptr) cudaFreeHost(sl.ptr);
    if (sl.ev) cudaEventDestroy(sl.ev);
  }
  delete P;
  return KV_OK;
}

kv_status_t kv_request_open(kv_pool_t* P, int32_t* req_id) {
  if (!P || !req_id) return fail(KV_ERR_INVALID_ARG, "kv_request_open: null argument");
  for (int32_t r = 0; r < P->cfg.max_requests; ++r)
    if (!P->reqs[r].open) {
      const uint64_t v = P->reqs[r].version;
      P->reqs[r] = Request();
      P->reqs[r].open = true;
      P->reqs[r].shape = ++P->shape_clock;
      P->reqs[r].version = v + 1;
      *req_id = r;
      return KV_OK;
    }
  return fail(KV_ERR_OOM, "kv_request_open: all %d request slots are open", P->cfg.max_requests);
}

kv_status_t kv_request_close(kv_pool_t* P, int32_t r) {
  if (!P || !req_ok(P, r)) return fail(KV_ERR_INVALID_ARG, "kv_request_close: request %d is not open", r);
  if (!P->hdead.empty()) {
    // the device words of freed pages are cleared before their ids return
    DeviceGuard dg(P->cfg.device);
    const int hkv = P->cfg.num_kv_heads;
    for (int32_t id : P->reqs[r].table) {
      uint32_t* w = &P->hdead[(size_t)id * hkv];
      if (std::any_of(w, w + hkv, [](uint32_t x) { return x != 0u; })) {
        std::fill(w, w + hkv, 0u);
        KV_CUDA(cudaMemsetAsync(P->d_hdead + (size_t)id * hkv, 0, (size_t)hkv * sizeof(uint32_t), P->last_stream));
      }
    }
  }
  for (int32_t id : P->reqs[r].table) {
    P->fill[id] = 0;
    P->live[id] = 0;
    free_list(P, id).insert(id);
  }
  if (!P->n_fp.empty()) P->n_fp[r] = 0;
  const uint64_t v = P->reqs[r].version;
  P->reqs[r] = Request();
  P->reqs[r].version = v + 1;
  return KV_OK;
}

kv_status_t kv_request_info(kv_pool_t* P, int32_t r, int32_t* n_pages, int64_t* n_tokens) {
  if (!P || !req_ok(P, r)) return fail(KV_ERR_INVALID_ARG, "kv_request_info: request %d is not open", r);
  if (n_pages) *n_pages = (int32_t)P->reqs[r].table.size();
  if (n_tokens) *n_tokens = (int64_t)P->reqs[r].loc.size();
  return KV_OK;
}

kv_status_t kv_set_decode_impl(kv_pool_t* P, int32_t impl) {
  if (!P || impl < KV_DECODE_AUTO || impl > KV_DECODE_MMA) return fail(KV_ERR_INVALID_ARG, "kv_set_decode_impl: bad impl");
  P->decode_impl = impl;
  return KV_OK;
}

kv_status_t kv_set_wait_limit(kv_pool_t* P, int64_t first_wait_spins) {
  if (!P) return fail(KV_ERR_INVALID_ARG, "kv_set_wait_limit: null pool");
  if (first_wait_spins < -1 || first_wait_spins > (int64_t)UINT32_MAX)
    return fail(KV_ERR_INVALID_ARG, "kv_set_wait_limit: first_wait_spins must be -1 or in [0, 2^32)");
  P->first_wait_spins = first_wait_spins;
  return KV_OK;
}

kv_status_t kv_pool_sync(kv_pool_t* P) {
  if (!P) return fail(KV_ERR_INVALID_ARG, "kv_pool_sync: null pool");
  DeviceGuard dg(P->cfg.device);
  if (P->last_stream) KV_CUDA(cudaStreamSynchronize(P->last_stream));
  KV_CUDA(cudaDeviceSynchronize());
  uint32_t st = 0;
  KV_CUDA(cudaMemcpy(&st, P->d_status, 4, cudaMemcpyDeviceToHost));
  if (st) KV_CUDA(cudaMemset(P->d_status, 0, 4));
  if (st & kStatusTimeout) return fail(KV_ERR_DEVICE_TIMEOUT, "kv_pool_sync: a bounded device wait expired");
  if (st & kStatusRange) return fail(KV_ERR_RANGE, "kv_pool_sync: an appended value was NaN, Inf or |x| > 65504");
  return KV_OK;
}

}  // extern "C"

extern "C" {

kv_status_t kv_append_quant(kv_pool_t* P, const void* k, const void* v, const int32_t* req_ids,
                            const uint8_t* bits, int64_t n_tok, void* stream) {
  if (!P) return fail(KV_ERR_INVALID_ARG, "kv_append_quant: null pool");
  if (n_tok < 0 || n_tok > INT32_MAX) return fail(KV_ERR_INVALID_ARG, "kv_append_quant: bad n_tok %lld", (long long)n_tok);
  if (n_tok == 0) return KV_OK;
  if (!k || !v || !req_ids || !bits) return fail(KV_ERR_INVALID_ARG, "kv_append_quant: null pointer");
  // Per-request state of this call, found through a pool-wide slot index.
  struct CallReq {
    int32_t r;
    int32_t old_len;       // table length before the call
    int32_t q_left;        // INT2-tagged tokens of r not yet routed in this call
    int32_t tail_job;      // append job of the current INT4 tail page (-1: none yet)
    int32_t tail3_job;     // append job of the current INT3 tail page (-1: none yet)
    int32_t tailf_job;     // append job of the current FP4 tail page (-1: none yet)
    int32_t stag_job;      // append job of the current staging page (-1: none / direct)
    bool stag_direct;      // the current staging page fills within this call: quantized directly to INT2
    int32_t ngrp;          // tokens collected for it so far
    int32_t grp[kPage];    // their token indices, in slot order
    // dry-run state
    bool tail; int tailfill; bool tail3; int tail3fill; bool tailf; int tailffill; bool stag; int stagfill;
    int64_t tablen;
    int64_t npos;          // the request's token positions after the call
  };
  std::vector<CallReq> cr;
  if (P->call_slot.size() != (size_t)P->cfg.max_requests) P->call_slot.assign((size_t)P->cfg.max_requests, -1);
  auto slot_of = [&](int32_t r) -> CallReq& {
    int32_t& sl = P->call_slot[(size_t)r];
    if (sl < 0) {
      const Request& R = P->reqs[r];
      sl = (int32_t)cr.size();
      CallReq c{};
      c.r = r;
      c.old_len = (int32_t)R.table.size();
      c.tail_job = c.tail3_job = c.tailf_job = c.stag_job = -1;
      c.tail = R.tail4 >= 0;
      c.tailfill = c.tail ? (int)P->fill[R.tail4] : 0;
      c.tail3 = R.tail3 >= 0;
      c.tail3fill = c.tail3 ? (int)P->fill[R.tail3] : 0;
      c.tailf = R.tailf >= 0;
      c.tailffill = c.tailf ? (int)P->fill[R.tailf] : 0;
      c.stag = R.staging >= 0;
      c.stagfill = c.stag ? (int)P->fill[R.staging] : 0;
      c.tablen = (int64_t)R.table.size();
      c.npos = (int64_t)R.loc.size();
      cr.push_back(c);
    }
    return cr[(size_t)sl];
  };
  struct ResetSlots {
    kv_pool* P;
    std::vector<CallReq>* cr;
    ~ResetSlots() { for (const auto& c : *cr) P->call_slot[(size_t)c.r] = -1; }
  } reset_slots{P, &cr};

  // Bulk path: the call's tokens come in runs, one per request (a prefill
  // chunk of one request, or one chunk of each of several requests): every
  // run at least one page of tokens, no request in two runs.  Within a run
  // the per-token rules reduce to whole groups: INT4 tokens fill the tail
  // page and new pages of 32; INT2 tokens fill the open staging page, then
  // groups of 32 that complete within the call (direct INT2 jobs), then one
  // partial staging page.  Runs are routed in call order, and page ids are
  // taken in the same token order as the per-token loop takes them, so both
  // paths give the same pool.
  struct BulkRun {
    int32_t r;
    int64_t t0, n;            // the call's tokens [t0, t0 + n)
    int64_t o4, n4, o2, n2;   // its entries in the call's INT4 / INT2 lists
    // routing, from the request's state before the call
    int64_t cap4, new4, e, ndirect, rem;
    int f4, s0;
    bool repack;
  };
  std::vector<BulkRun> runs;
  bool bulk = n_tok >= kPage;
  // the call's INT4 / INT2 token indices, in order: the first n4 / n2
  // entries of scratch lists that only grow (no per-call clearing or filling)
  std::vector<int32_t>& i4 = P->scr_i4;
  std::vector<int32_t>& i2 = P->scr_i2;
  int64_t n4 = 0, n2 = 0;
  if (bulk) {
    // one pass: bits valid, run boundaries; raw pointers and local counts
    // (stores through vectors next to uint8_t loads defeat registers)
    if (i4.size() < (size_t)n_tok) i4.resize((size_t)n_tok);
    if (i2.size() < (size_t)n_tok) i2.resize((size_t)n_tok);
    int32_t* p4 = i4.data();
    int32_t* p2 = i2.data();
    int64_t c4 = 0, c2 = 0, changes = 0;
    int32_t rp = req_ids[0];
    bool ok = true;
    for (int64_t t = 0; t < n_tok; ++t) {
      const uint32_t b = bits[t];
      const int32_t rt = req_ids[t];
      ok &= (b == 2u) | (b == 4u);
      changes += rt != rp;
      rp = rt;
      p4[c4] = (int32_t)t;
      p2[c2] = (int32_t)t;
      c4 += b == 4u;
      c2 += b != 4u;
    }
    if (changes == 0) {
      runs.push_back(BulkRun{req_ids[0], 0, n_tok, 0, c4, 0, c2, 0, 0, 0, 0, 0, 0, 0, false});
    } else if (ok) {
      // several requests: a second pass finds the runs (this keeps the first
      // pass free of branches and calls)
      int64_t tb = 0, d4 = 0, d2 = 0, b4 = 0, b2 = 0;
      for (int64_t t = 1; t <= n_tok; ++t) {
        d4 += bits[t - 1] == 4u;
        d2 += bits[t - 1] != 4u;
        if (t == n_tok || req_ids[t] != req_ids[t - 1]) {
          runs.push_back(BulkRun{req_ids[tb], tb, t - tb, b4, d4 - b4, b2, d2 - b2, 0, 0, 0, 0, 0, 0, 0, false});
          tb = t;
          b4 = d4;
          b2 = d2;
        }
      }
    }
    // each run an open request of its own, at least a page of tokens long
    // (anything else: the per-token path, which also reports any error)
    for (const auto& u : runs) {
      if (!ok || u.n < kPage || !req_ok(P, u.r) || P->call_slot[(size_t)u.r] >= 0) {
        ok = false;
        break;
      }
      slot_of(u.r);
    }
    bulk = ok;
    n4 = c4;
    n2 = c2;
  }
  if (bulk) {
    int64_t need4 = 0, need2 = 0;
    for (auto& u : runs) {
      const Request& R = P->reqs[u.r];
      const bool tail_open = R.tail4 >= 0 && P->fill[R.tail4] < kPage;
      u.f4 = tail_open ? (int)P->fill[R.tail4] : 0;
      u.cap4 = tail_open ? std::min<int64_t>(u.n4, kPage - u.f4) : 0;
      u.new4 = (u.n4 - u.cap4 + kPage - 1) / kPage;
      u.s0 = R.staging >= 0 ? (int)P->fill[R.staging] : 0;
      u.e = R.staging >= 0 ? std::min<int64_t>(u.n2, kPage - u.s0) : 0;
      u.repack = R.staging >= 0 && u.s0 + u.e == kPage;
      u.ndirect = (u.n2 - u.e) / kPage;
      u.rem = (u.n2 - u.e) % kPage;
      const int64_t opens = u.new4 + u.ndirect + (u.rem > 0 ? 1 : 0);
      need4 += opens;
      need2 += u.ndirect + (u.repack ? 1 : 0);
      if ((int64_t)R.table.size() + opens > P->cfg.max_pages_per_request)
        return fail(KV_ERR_OOM, "kv_append_quant: request %d would exceed %d table entries", u.r,
                    P->cfg.max_pages_per_request);
      if ((int64_t)R.loc.size() + u.n > kMaxPositions)
        return fail(KV_ERR_INVALID_ARG, "kv_append_quant: request %d would exceed %lld token positions", u.r,
                    (long long)kMaxPositions);
    }
    if (need4 > (int64_t)P->free4.size() || need2 > (int64_t)P->free2.size())
      return fail(KV_ERR_OOM, "kv_append_quant: needs %lld INT4 + %lld INT2 pages, %zu + %zu free", (long long)need4,
                  (long long)need2, P->free4.size(), P->free2.size());
  }
  // Dry run: pages taken and table growth, so that OOM changes nothing.
  if (!bulk) {
    int64_t need4 = 0, need3 = 0, needf = 0, need2 = 0;
    for (int64_t t = 0; t < n_tok; ++t) {
      if (!req_ok(P, req_ids[t]))
        return fail(KV_ERR_INVALID_ARG, "kv_append_quant: token %lld: request %d not open", (long long)t, req_ids[t]);
      if ((bits[t] < 2 || bits[t] > 4) && bits[t] != KV_WIDTH_FP4)
        return fail(KV_ERR_INVALID_ARG, "kv_append_quant: token %lld: bits must be 2, 3, 4 or KV_WIDTH_FP4",
                    (long long)t);
      CallReq& c = slot_of(req_ids[t]);
      if (bits[t] == 4) {
        if (!c.tail || c.tailfill == kPage) { ++need4; ++c.tablen; c.tail = true; c.tailfill = 0; }
        ++c.tailfill;
      } else if (bits[t] == 3) {
        if (!c.tail3 || c.tail3fill == kPage) { ++need3; ++c.tablen; c.tail3 = true; c.tail3fill = 0; }
        ++c.tail3fill;
      } else if (bits[t] == KV_WIDTH_FP4) {
        if (!c.tailf || c.tailffill == kPage) { ++needf; ++c.tablen; c.tailf = true; c.tailffill = 0; }
        ++c.tailffill;
      } else {
        ++c.q_left;
        if (!c.stag) { ++need4; ++c.tablen; c.stag = true; c.stagfill = 0; }
        if (++c.stagfill == kPage) { ++need2; c.stag = false; }
      }
      if (c.tablen > P->cfg.max_pages_per_request)
        return fail(KV_ERR_OOM, "kv_append_quant: request %d would exceed %d table entries", req_ids[t], P->cfg.max_pages_per_request);
      if (++c.npos > kMaxPositions)
        return fail(KV_ERR_INVALID_ARG, "kv_append_quant: request %d would exceed %lld token positions", req_ids[t],
                    (long long)kMaxPositions);
    }
    if (need4 > (int64_t)P->free4.size() || need2 > (int64_t)P->free2.size())
      return fail(KV_ERR_OOM, "kv_append_quant: needs %lld INT4 + %lld INT2 pages, %zu + %zu free", (long long)need4,
                  (long long)need2, P->free4.size(), P->free2.size());
    if (need3 > (int64_t)P->free3.size())
      return fail(KV_ERR_OOM, "kv_append_quant: needs %lld INT3 pages, %zu free", (long long)need3, P->free3.size());
    if (needf > (int64_t)P->freef.size())
      return fail(KV_ERR_OOM, "kv_append_quant: needs %lld FP4 pages, %zu free", (long long)needf, P->freef.size());
  }
  // room for this call's tokens in each position map; growth is geometric
  // (reserving just the new size on every call would copy the whole map)
  for (const auto& c : cr) {
    Request& R = P->reqs[c.r];
    const size_t need = R.loc.size() + (size_t)n_tok;
    if (R.loc.capacity() < need) R.loc.reserve(std::max(need, 2 * R.loc.capacity()));
  }
  DeviceGuard dg(P->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  kv_status_t st = order_after_previous(P, s);
  if (st != KV_OK) return st;

  // Routing in token order (page ids are taken exactly as the per-token rules
  // dictate).  A staging page that starts empty and is filled within this
  // call is never materialised: its 32 tokens go to a direct job that
  // quantizes them to INT4, dequantizes and requantizes to INT2 in one kernel
  // (the same values the staging page and its repack would give).
  std::vector<AppendJob> jobs;
  std::vector<int32_t> job_req;                        // request of each job
  std::vector<RepackJob> repacks;
  std::vector<DirectJob> directs;
  std::vector<int32_t>& dtoks = P->scr_dtoks;          // 32 token indices per direct job
  std::vector<int32_t>& toks = P->scr_toks;            // token indices of the append jobs, job by job in slot order
  dtoks.clear();
  toks.clear();
  std::vector<int32_t> deferred;
  Dirty dirty;   // table rewrites the append kernel does not cover (repacks)
  std::vector<TableUpd> hupd;   // per-head exclusion words carried by repacks / cleared by frees
  int64_t bulk_job_toks = 0;    // bulk path: tokens of the append jobs
  if (bulk) {
  for (const BulkRun& u : runs) {
    const int32_t r = u.r;
    Request& R = P->reqs[r];
    const int32_t* const l4 = i4.data() + u.o4;   // the run's INT4 / INT2 tokens (call indices)
    const int32_t* const l2 = i2.data() + u.o2;
    const int64_t T0 = (int64_t)R.loc.size();
    const int64_t P0 = T0 - u.t0;                 // the request's position of call token t: P0 + t
    R.loc.resize((size_t)(T0 + u.n));   // every new entry is written below
    auto put = [&](int32_t page, int slot, int32_t t) {
      P->pos[(size_t)page * kPage + slot] = (int32_t)(P0 + t);
      R.loc[(size_t)(P0 + t)] = ((uint32_t)page << 5) | (uint32_t)slot;
    };
    auto slots = [](int first, int64_t n) { return (uint32_t)((n >= kPage ? 0xFFFFFFFFull : ((1ull << n) - 1)) << first); };
    // An append job over the run's INT4 (int4_list) or INT2 tokens
    // [a, a + n) into slots first .. of page.  Its tok_off indexes the call's
    // two lists as if the INT2 list followed the n4 INT4 entries; the upload
    // below places the lists and adjusts the offsets into the INT2 list.
    int32_t* const pos = P->pos.data();
    uint32_t* const loc = R.loc.data();
    auto add_job = [&](int32_t page, int first, bool int4_list, int64_t a, int64_t n) {
      const int64_t off = (int4_list ? u.o4 : n4 + u.o2) + a;
      jobs.push_back(AppendJob{page, first, (int32_t)n, (int32_t)off, -1, 0u, -1, 0});
      job_req.push_back(r);
      const int32_t* src = (int4_list ? l4 : l2) + a;
      int32_t* pp = pos + (size_t)page * kPage + first;
      const uint32_t base = ((uint32_t)page << 5) | (uint32_t)first;
      for (int64_t q = 0; q < n; ++q) {
        const int32_t t = src[q];
        pp[q] = (int32_t)(P0 + t);
        loc[P0 + t] = base + (uint32_t)q;
      }
      bulk_job_toks += n;
      P->fill[page] = (uint8_t)(first + n);
      P->live[page] |= slots(first, n);
    };
    // INT4 pages and staging pages take ids in the token order of their
    // first token; INT2 pages in the order their groups complete
    std::vector<int32_t> id4((size_t)u.new4), idS((size_t)(u.ndirect + (u.rem > 0 ? 1 : 0)));
    {
      size_t a = 0, b = 0;
      while (a < id4.size() || b < idS.size()) {
        const int32_t ta = a < id4.size() ? l4[(size_t)(u.cap4 + kPage * (int64_t)a)] : INT32_MAX;
        const int32_t tb = b < idS.size() ? l2[(size_t)(u.e + kPage * (int64_t)b)] : INT32_MAX;
        if (ta < tb) id4[a++] = P->free4.take_lowest();
        else idS[b++] = P->free4.take_lowest();
      }
    }
    const int32_t nid_rep = u.repack ? P->free2.take_lowest() : -1;
    std::vector<int32_t> idD((size_t)u.ndirect);
    for (auto& x : idD) x = P->free2.take_lowest();
    // table entries appended in this call, with the token that appends them
    std::vector<std::pair<int32_t, int32_t>> app;   // (token, page id)
    // INT4: the open tail page, then new pages
    if (u.cap4 > 0) add_job(R.tail4, u.f4, true, 0, u.cap4);
    for (int64_t q = 0; q < u.new4; ++q) {
      const int64_t a = u.cap4 + kPage * q;
      const int32_t pg = id4[(size_t)q];
      P->fill[pg] = 0;
      P->live[pg] = 0u;
      add_job(pg, 0, true, a, std::min<int64_t>(kPage, u.n4 - a));
      app.emplace_back(l4[(size_t)a], pg);
    }
    if (u.new4 > 0) R.tail4 = id4[(size_t)(u.new4 - 1)];
    // INT2: the open staging page
    if (u.e > 0) add_job(R.staging, u.s0, false, 0, u.e);
    if (u.repack) {
      const int32_t sp = R.staging;
      P->fill[nid_rep] = kPage;
      P->live[nid_rep] = P->live[sp];
      hdead_copy(P, nid_rep, sp, hupd);
      for (int sl = 0; sl < kPage; ++sl) {
        const int32_t pp = P->pos[(size_t)sp * kPage + sl];
        P->pos[(size_t)nid_rep * kPage + sl] = pp;
        R.loc[(size_t)pp] = ((uint32_t)nid_rep << 5) | (uint32_t)sl;
      }
      const auto rit = std::find(R.table.rbegin(), R.table.rend(), sp);
      const auto it = std::next(rit).base();
      dirty.structural(r, (int32_t)(it - R.table.begin()));
      R.table.erase(it);
      R.shape = ++P->shape_clock;
      repacks.push_back(RepackJob{sp, nid_rep});
      deferred.push_back(sp);
      app.emplace_back(l2[(size_t)(u.e - 1)], nid_rep);
      R.staging = -1;
    }
    // groups of 32 completed in this call: direct INT2 jobs (their staging
    // ids are taken and freed, as the per-token path does)
    for (int64_t g = 0; g < u.ndirect; ++g) {
      const int64_t a = u.e + kPage * g;
      const int32_t sg = idS[(size_t)g], nid = idD[(size_t)g];
      for (int sl = 0; sl < kPage; ++sl) put(nid, sl, l2[(size_t)(a + sl)]);
      P->fill[sg] = kPage;
      P->live[sg] = 0xFFFFFFFFu;
      P->fill[nid] = kPage;
      P->live[nid] = 0xFFFFFFFFu;
      directs.push_back(DirectJob{nid, (int32_t)(u.o2 + a)});   // its tokens: the INT2 list, uploaded whole
      deferred.push_back(sg);
      app.emplace_back(l2[(size_t)(a + kPage - 1)], nid);
    }
    if (u.ndirect > 0 && !u.repack) dirty.structural(r, (int32_t)R.table.size());
    // the last, partial staging page
    if (u.rem > 0) {
      const int64_t a = u.e + kPage * u.ndirect;
      const int32_t sp = idS[(size_t)u.ndirect];
      P->fill[sp] = 0;
      P->live[sp] = 0u;
      add_job(sp, 0, false, a, u.rem);
      app.emplace_back(l2[(size_t)a], sp);
      R.staging = sp;
    }
    std::sort(app.begin(), app.end());
    for (const auto& x : app) R.table.push_back(x.second);
    if (!app.empty() || u.repack) ++R.version;
  }
  } else {
  std::vector<int32_t> tok_job((size_t)n_tok, -1), tok_slot((size_t)n_tok);
  for (int64_t t = 0; t < n_tok; ++t) {
    const int32_t r = req_ids[t];
    Request& R = P->reqs[r];
    CallReq& c = cr[(size_t)P->call_slot[(size_t)r]];
    const int64_t pos = (int64_t)R.loc.size();
    const bool b4 = bits[t] == 4, b3 = bits[t] == 3, bf = bits[t] == KV_WIDTH_FP4;
    // INT4 tokens fill the INT4 tail, INT3 and FP4 tokens their own tails, INT2 tokens the (INT4) staging page
    int32_t& cur = b4 ? R.tail4 : (b3 ? R.tail3 : (bf ? R.tailf : R.staging));
    if (cur < 0 || P->fill[cur] == kPage) {
      cur = (b3 ? P->free3 : (bf ? P->freef : P->free4)).take_lowest();
      P->fill[cur] = 0;
      P->live[cur] = 0;
      R.table.push_back(cur);
      ++R.version;
      if (b4) {
        c.tail_job = -1;
      } else if (b3) {
        c.tail3_job = -1;
      } else if (bf) {
        c.tailf_job = -1;
      } else {
        c.stag_job = -1;
        c.stag_direct = c.q_left >= kPage;
        c.ngrp = 0;
      }
    }
    const int slot = P->fill[cur]++;
    P->live[cur] |= 1u << slot;
    P->pos[(size_t)cur * kPage + slot] = (int32_t)pos;
    R.loc.push_back(((uint32_t)cur << 5) | (uint32_t)slot);
    const bool b2 = !b4 && !b3 && !bf;
    if (b2) --c.q_left;
    if (b2 && c.stag_direct) {
      c.grp[c.ngrp++] = (int32_t)t;
    } else {
      int32_t& jb = b4 ? c.tail_job : (b3 ? c.tail3_job : (bf ? c.tailf_job : c.stag_job));
      if (jb < 0) {
        jb = (int32_t)jobs.size();
        jobs.push_back(AppendJob{cur, slot, 0, 0, -1, 0u, -1, 0});
        job_req.push_back(r);
      }
      ++jobs[(size_t)jb].n_slots;
      tok_job[t] = jb;
      tok_slot[t] = slot;
    }
    if (b2 && P->fill[cur] == kPage) {
      // 32 qualifying tokens: requantize the staging page into a new INT2 page.
      const int32_t nid = P->free2.take_lowest();
      P->fill[nid] = kPage;
      P->live[nid] = P->live[cur];
      hdead_copy(P, nid, cur, hupd);
      for (int sl = 0; sl < kPage; ++sl) {
        const int32_t p = P->pos[(size_t)cur * kPage + sl];
        P->pos[(size_t)nid * kPage + sl] = p;
        R.loc[p] = ((uint32_t)nid << 5) | (uint32_t)sl;
      }
      const auto rit = std::find(R.table.rbegin(), R.table.rend(), cur);   // the staging page sits near the end
      const auto it = std::next(rit).base();
      dirty.structural(r, (int32_t)(it - R.table.begin()));
      R.table.erase(it);
      R.shape = ++P->shape_clock;
      R.table.push_back(nid);
      if (c.stag_direct) {
        directs.push_back(DirectJob{nid, (int32_t)dtoks.size()});
        dtoks.insert(dtoks.end(), c.grp, c.grp + kPage);
        c.ngrp = 0;
      } else {
        repacks.push_back(RepackJob{cur, nid});
      }
      deferred.push_back(cur);
      cur = -1;
      c.stag_job = -1;
      c.stag_direct = false;
      ++R.version;
    }
  }
  int32_t off = 0;
  for (auto& j : jobs) { j.tok_off = off; off += j.n_slots; }
  toks.assign((size_t)off, 0);
  for (int64_t t = 0; t < n_tok; ++t) {
    if (tok_job[t] < 0) continue;   // routed to a direct job
    const AppendJob& j = jobs[(size_t)tok_job[t]];
    toks[(size_t)(j.tok_off + (tok_slot[t] - j.first_slot))] = (int32_t)t;
  }
  }   // per-token path
  const int64_t off = bulk ? bulk_job_toks : (int64_t)toks.size();
  for (int32_t id : deferred) {
    P->fill[id] = 0;
    P->live[id] = 0;
    hdead_clear(P, id, hupd);
    P->free4.insert(id);
  }
  // Table entries the append kernel writes: each job's page where it sits in
  // the final table (pages added at the end or filled in place), and the
  // final table length of every request that grew.
  const uint32_t mp = (uint32_t)P->cfg.max_pages_per_request;
  {
    // A job's page is in its request's final table unless a repack removed it
    // (freed above, fill 0).  Appended pages sit near the end of the table, so
    // one backward scan per request finds them all.
    if (P->page_job.size() != P->fill.size()) P->page_job.assign(P->fill.size(), -1);
    std::vector<int32_t> need(cr.size(), 0);
    for (size_t j = 0; j < jobs.size(); ++j) {
      AppendJob& J = jobs[j];
      const int32_t r = job_req[j];
      const int32_t ci = P->call_slot[(size_t)r];
      const int32_t len = (int32_t)P->reqs[r].table.size();
      if (len != cr[(size_t)ci].old_len) {
        J.ntab_req = r;
        J.ntab_len = len;
      }
      if (P->fill[J.page] > 0) {
        P->page_job[(size_t)J.page] = (int32_t)j;
        J.live = P->live[J.page];
        ++need[(size_t)ci];
      }
    }
    for (size_t ci = 0; ci < cr.size(); ++ci) {
      const int32_t r = cr[ci].r;
      const auto& tb = P->reqs[r].table;
      for (int32_t i = (int32_t)tb.size() - 1; i >= 0 && need[ci] > 0; --i) {
        const int32_t j = P->page_job[(size_t)tb[i]];
        if (j >= 0 && job_req[(size_t)j] == r) {
          jobs[(size_t)j].tab_index = (int32_t)(r * mp + (uint32_t)i);
          --need[ci];
        }
      }
    }
    for (const auto& J : jobs) P->page_job[(size_t)J.page] = -1;
  }
  std::vector<TableUpd> upd;
  emit_updates(P, dirty, upd);
  hdead_final(P, hupd);
  upd.insert(upd.end(), hupd.begin(), hupd.end());

  // INT3 and FP4 jobs go last (INT3, then FP4), to their own kernels
  size_t n_i3 = 0, n_f4 = 0;
  for (const auto& j : jobs) {
    n_i3 += is_int3(P, j.page) ? 1 : 0;
    n_f4 += is_fp4(P, j.page) ? 1 : 0;
  }
  if (n_i3 + n_f4) {
    std::stable_partition(jobs.begin(), jobs.end(), [&](const AppendJob& j) { return width_of(P, j.page) == 2 ||
                                                                                      width_of(P, j.page) == 4; });
    std::stable_partition(jobs.end() - (ptrdiff_t)(n_i3 + n_f4), jobs.end(),
                          [&](const AppendJob& j) { return is_int3(P, j.page); });
  }
  const bool small = n_i3 + n_f4 == 0 && jobs.size() <= (size_t)SmallAppend::kMaxJobs && off <= SmallAppend::kMaxToks;
  // Large calls with 16-byte aligned K/V rows: fresh pages filled with 32
  // tokens go to the bulk INT4 kernel, direct groups to the bulk INT2 kernel.
  const bool aligned = ((uintptr_t)k % 16 == 0) && ((uintptr_t)v % 16 == 0);
  const bool use_bulk = !small && aligned;
  size_t n_full = 0;
  const auto jobs4_end = jobs.end() - (ptrdiff_t)(n_i3 + n_f4);
  if (use_bulk) {
    std::stable_partition(jobs.begin(), jobs4_end, [](const AppendJob& j) { return !(j.first_slot == 0 && j.n_slots == kPage); });
    for (auto it = jobs.begin(); it != jobs4_end; ++it) n_full += (it->first_slot == 0 && it->n_slots == kPage) ? 1 : 0;
  }
  if (bulk && small) {
    // the small launch carries its token lists by value: gather each job's tokens
    toks.clear();
    for (auto& j : jobs) {
      const int32_t* src = j.tok_off < n4 ? i4.data() + j.tok_off : i2.data() + (j.tok_off - n4);
      j.tok_off = (int32_t)toks.size();
      toks.insert(toks.end(), src, src + j.n_slots);
    }
  }
  Upload u;
  const size_t o_jobs = small ? 0 : u.add(jobs.data(), jobs.size() * sizeof(AppendJob));
  size_t o_toks = 0, o_dtok = 0;
  if (bulk) {
    // the call's INT4 and INT2 token lists as they are: the append jobs index
    // both, the direct INT2 jobs the INT2 list
    o_toks = small ? 0 : u.add(i4.data(), (size_t)n4 * sizeof(int32_t));
    o_dtok = u.add(i2.data(), (size_t)n2 * sizeof(int32_t));
    if (!small) {
      const int64_t shift = (int64_t)(o_dtok - o_toks) / (int64_t)sizeof(int32_t) - n4;
      for (auto& j : jobs)
        if (j.tok_off >= n4) j.tok_off = (int32_t)(j.tok_off + shift);
    }
  } else {
    o_toks = small ? 0 : u.add(toks.data(), toks.size() * sizeof(int32_t));
    o_dtok = u.add(dtoks.data(), dtoks.size() * sizeof(int32_t));
  }
  const size_t o_rep = u.add(repacks.data(), repacks.size() * sizeof(RepackJob));
  const size_t o_dir = u.add(directs.data(), directs.size() * sizeof(DirectJob));
  const size_t o_upd = u.add(upd.data(), upd.size() * sizeof(TableUpd));
  if ((st = upload(P, u, s)) != KV_OK) return st;
  uint8_t* base = (uint8_t*)P->upload.ptr;
  if (small) {
    SmallAppend sa;
    std::copy(jobs.begin(), jobs.end(), sa.jobs);
    std::copy(toks.begin(), toks.end(), sa.toks);
    KV_CUDA(launch_append(P, k, v, nullptr, (int)jobs.size(), nullptr, &sa, s));
  } else {
    const int n_part = (int)(jobs.size() - n_i3 - n_f4 - n_full);
    KV_CUDA(launch_append(P, k, v, (const AppendJob*)(base + o_jobs), n_part, (const int32_t*)(base + o_toks),
                          nullptr, s));
    if (n_full)
      KV_CUDA(launch_bulk_int4(P, k, v, (const AppendJob*)(base + o_jobs) + n_part, (int)n_full,
                               (const int32_t*)(base + o_toks), s));
    if (n_i3)
      KV_CUDA(launch_append_int3(P, k, v, (const AppendJob*)(base + o_jobs) + (jobs.size() - n_i3 - n_f4),
                                 (int)n_i3, (const int32_t*)(base + o_toks), s));
    if (n_f4)
      KV_CUDA(launch_append_fp4(P, k, v, (const AppendJob*)(base + o_jobs) + (jobs.size() - n_f4), (int)n_f4,
                                (const int32_t*)(base + o_toks), s));
  }
  if (use_bulk)
    KV_CUDA(launch_bulk_int2(P, k, v, (const DirectJob*)(base + o_dir), (int)directs.size(),
                             (const int32_t*)(base + o_dtok), s));
  else
    KV_CUDA(launch_direct_int2(P, k, v, (const DirectJob*)(base + o_dir), (int)directs.size(),
                               (const int32_t*)(base + o_dtok), s));
  KV_CUDA(launch_repack(P, (const RepackJob*)(base + o_rep), (int)repacks.size(), s));
  KV_CUDA(launch_scatter(P, (const TableUpd*)(base + o_upd), (int)upd.size(), s));
  return KV_OK;
}

kv_status_t kv_reorder_pages(kv_pool_t* P, const int32_t* req_ids, int32_t n_req, void* stream) {
  if (!P || n_req < 0 || (n_req > 0 && !req_ids)) return fail(KV_ERR_INVALID_ARG, "kv_reorder_pages: bad arguments");
  for (int32_t i = 0; i < n_req; ++i)
    if (!req_ok(P, req_ids[i])) return fail(KV_ERR_INVALID_ARG, "kv_reorder_pages: request %d not open", req_ids[i]);
  Dirty dirty;
  for (int32_t i = 0; i < n_req; ++i) {
    Request& R = P->reqs[req_ids[i]];
    if (R.ordered_version == R.version) continue;   // unchanged since it was last found INT2-first
    if (P->cfg.n_int3_pages > 0 || P->cfg.n_fp4_pages > 0) {
      // more widths: a stable sort by width (INT2, INT3, INT4, FP4)
      auto by_width = [&](int32_t a, int32_t b) { return width_of(P, a) < width_of(P, b); };
      if (!std::is_sorted(R.table.begin(), R.table.end(), by_width)) {
        std::vector<int32_t> old = R.table;
        std::stable_sort(R.table.begin(), R.table.end(), by_width);
        int32_t from = 0;
        while (old[(size_t)from] == R.table[(size_t)from]) ++from;
        R.shape = ++P->shape_clock;
        dirty.structural(req_ids[i], from);
        ++R.version;
      }
      R.ordered_version = R.version;
      continue;
    }
    auto first_int4 = std::find_if(R.table.begin(), R.table.end(), [&](int32_t id) { return !is_int2(P, id); });
    if (std::find_if(first_int4, R.table.end(), [&](int32_t id) { return is_int2(P, id); }) != R.table.end()) {
      const int32_t from = (int32_t)(first_int4 - R.table.begin());
      std::stable_partition(R.table.begin(), R.table.end(), [&](int32_t id) { return is_int2(P, id); });
      R.shape = ++P->shape_clock;
      dirty.structural(req_ids[i], from);
      ++R.version;
    }
    R.ordered_version = R.version;
  }
  if (dirty.from.empty()) return KV_OK;
  DeviceGuard dg(P->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  kv_status_t st = order_after_previous(P, s);
  if (st != KV_OK) return st;
  std::vector<TableUpd> upd;
  emit_updates(P, dirty, upd);
  Upload u;
  const size_t o = u.add(upd.data(), upd.size() * sizeof(TableUpd));
  if ((st = upload(P, u, s)) != KV_OK) return st;
  KV_CUDA(launch_scatter(P, (const TableUpd*)((uint8_t*)P->upload.ptr + o), (int)upd.size(), s));
  return KV_OK;
}

kv_status_t kv_evict_slots(kv_pool_t* P, const int32_t* req_ids, const int64_t* token_pos, int64_t n, void* stream) {
  if (!P || n < 0 || (n > 0 && (!req_ids || !token_pos))) return fail(KV_ERR_INVALID_ARG, "kv_evict_slots: bad arguments");
  for (int64_t i = 0; i < n; ++i) {
    if (!req_ok(P, req_ids[i])) return fail(KV_ERR_INVALID_ARG, "kv_evict_slots: request %d not open", req_ids[i]);
    if (token_pos[i] < 0 || token_pos[i] >= (int64_t)P->reqs[req_ids[i]].loc.size())
      return fail(KV_ERR_INVALID_ARG, "kv_evict_slots: position %lld out of range", (long long)token_pos[i]);
  }
  Dirty dirty;
  bool any = false;
  for (int64_t i = 0; i < n; ++i) {
    const uint32_t l = P->reqs[req_ids[i]].loc[token_pos[i]];
    if (l == kDroppedLoc) continue;   // its page was dropped: already dead
    const int32_t id = (int32_t)(l >> 5);
    const uint32_t bit = 1u << (l & 31u);
    if (P->live[id] & bit) {
      P->live[id] &= ~bit;
      dirty.live(req_ids[i], id);
      any = true;
    }
  }
  if (!any) return KV_OK;
  DeviceGuard dg(P->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  kv_status_t st = order_after_previous(P, s);
  if (st != KV_OK) return st;
  std::vector<TableUpd> upd;
  emit_updates(P, dirty, upd);
  Upload u;
  const size_t o = u.add(upd.data(), upd.size() * sizeof(TableUpd));
  if ((st = upload(P, u, s)) != KV_OK) return st;
  KV_CUDA(launch_scatter(P, (const TableUpd*)((uint8_t*)P->upload.ptr + o), (int)upd.size(), s));
  return KV_OK;
}

kv_status_t kv_evict_slots_head(kv_pool_t* P, const int32_t* req_ids, const int64_t* token_pos,
                                const int32_t* kv_heads, int64_t n, void* stream) {
  if (!P || n < 0 || (n > 0 && (!req_ids || !token_pos || !kv_heads)))
    return fail(KV_ERR_INVALID_ARG, "kv_evict_slots_head: bad arguments");
  const int hkv = P->cfg.num_kv_heads;
  for (int64_t i = 0; i < n; ++i) {
    if (!req_ok(P, req_ids[i])) return fail(KV_ERR_INVALID_ARG, "kv_evict_slots_head: request %d not open", req_ids[i]);
    if (token_pos[i] < 0 || token_pos[i] >= (int64_t)P->reqs[req_ids[i]].loc.size())
      return fail(KV_ERR_INVALID_ARG, "kv_evict_slots_head: position %lld out of range", (long long)token_pos[i]);
    if (kv_heads[i] < 0 || kv_heads[i] >= hkv)
      return fail(KV_ERR_INVALID_ARG, "kv_evict_slots_head: kv head %d out of range", kv_heads[i]);
  }
  if (n == 0) return KV_OK;
  DeviceGuard dg(P->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  kv_status_t st = order_after_previous(P, s);
  if (st != KV_OK) return st;
  if (P->hdead.empty()) {
    // first use: one exclusion word per (page id, kv head), all clear
    const size_t words = P->fill.size() * (size_t)hkv;
    if (cudaMalloc(&P->d_hdead, words * sizeof(uint32_t)) != cudaSuccess) {
      cudaGetLastError();
      P->d_hdead = nullptr;
      return fail(KV_ERR_OOM, "kv_evict_slots_head: cannot allocate %zu exclusion words", words);
    }
    KV_CUDA(cudaMemsetAsync(P->d_hdead, 0, words * sizeof(uint32_t), s));
    try {
      P->hdead.assign(words, 0u);
    } catch (...) {
      cudaFree(P->d_hdead);
      P->d_hdead = nullptr;
      return fail(KV_ERR_OOM, "kv_evict_slots_head: host allocation failed");
    }
  }
  std::vector<TableUpd> upd;
  for (int64_t i = 0; i < n; ++i) {
    const uint32_t l = P->reqs[req_ids[i]].loc[token_pos[i]];
    if (l == kDroppedLoc) continue;   // its page was dropped: already dead for every head
    const int32_t id = (int32_t)(l >> 5);
    hdead_set(P, id, kv_heads[i], P->hdead[(size_t)id * hkv + kv_heads[i]] | (1u << (l & 31u)), upd);
  }
  if (upd.empty()) return KV_OK;
  P->plan_impl = -1;   // page costs per head changed: plan again at the next decode
  hdead_final(P, upd);
  Upload u;
  const size_t o = u.add(upd.data(), upd.size() * sizeof(TableUpd));
  if ((st = upload(P, u, s)) != KV_OK) return st;
  KV_CUDA(launch_scatter(P, (const TableUpd*)((uint8_t*)P->upload.ptr + o), (int)upd.size(), s));
  return KV_OK;
}

kv_status_t kv_drop_dead_pages(kv_pool_t* P, const int32_t* req_ids, int32_t n_req, void* stream) {
  if (!P || n_req < 0 || (n_req > 0 && !req_ids)) return fail(KV_ERR_INVALID_ARG, "kv_drop_dead_pages: bad arguments");
  for (int32_t i = 0; i < n_req; ++i)
    if (!req_ok(P, req_ids[i])) return fail(KV_ERR_INVALID_ARG, "kv_drop_dead_pages: request %d not open", req_ids[i]);
  const int hkv = P->cfg.num_kv_heads;
  Dirty dirty;
  std::vector<TableUpd> hupd;
  for (int32_t q = 0; q < n_req; ++q) {
    const int32_t r = req_ids[q];
    Request& R = P->reqs[r];
    int32_t first = -1;
    size_t w = 0;
    for (size_t i = 0; i < R.table.size(); ++i) {
      const int32_t id = R.table[i];
      bool dead = P->fill[id] == kPage;
      if (dead) {
        if (P->hdead.empty()) {
          dead = P->live[id] == 0u;
        } else {
          for (int h = 0; h < hkv && dead; ++h) dead = (P->live[id] & ~P->hdead[(size_t)id * hkv + h]) == 0u;
        }
      }
      if (!dead) {
        R.table[w++] = id;
        continue;
      }
      if (first < 0) first = (int32_t)i;
      for (int sl = 0; sl < kPage; ++sl) {
        const int32_t pp = P->pos[(size_t)id * kPage + sl];
        if (pp >= 0 && (size_t)pp < R.loc.size()) R.loc[(size_t)pp] = kDroppedLoc;
      }
      if (R.tail4 == id) R.tail4 = -1;
      if (R.tail3 == id) R.tail3 = -1;
      if (R.tailf == id) R.tailf = -1;
      if (R.staging == id) R.staging = -1;
      P->fill[id] = 0;
      P->live[id] = 0u;
      hdead_clear(P, id, hupd);
      free_list(P, id).insert(id);
    }
    if (first < 0) continue;
    R.table.resize(w);
    ++R.version;
    R.shape = ++P->shape_clock;
    dirty.structural(r, first);
  }
  if (dirty.from.empty()) return KV_OK;
  DeviceGuard dg(P->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  kv_status_t st = order_after_previous(P, s);
  if (st != KV_OK) return st;
  std::vector<TableUpd> upd;
  emit_updates(P, dirty, upd);
  hdead_final(P, hupd);
  upd.insert(upd.end(), hupd.begin(), hupd.end());
  Upload u;
  const size_t o = u.add(upd.data(), upd.size() * sizeof(TableUpd));
  if ((st = upload(P, u, s)) != KV_OK) return st;
  KV_CUDA(launch_scatter(P, (const TableUpd*)((uint8_t*)P->upload.ptr + o), (int)upd.size(), s));
  return KV_OK;
}

kv_status_t kv_fp_configure(kv_pool_t* P, int32_t max_tokens) {
  if (!P || max_tokens < 0) return fail(KV_ERR_INVALID_ARG, "kv_fp_configure: bad arguments");
  for (int32_t x : P->n_fp)
    if (x > 0) return fail(KV_ERR_INVALID_ARG, "kv_fp_configure: a full-precision list is not empty");
  DeviceGuard dg(P->cfg.device);
  if (P->last_stream) KV_CUDA(cudaStreamSynchronize(P->last_stream));
  KV_CUDA(cudaDeviceSynchronize());
  cudaFree(P->d_fpk);
  cudaFree(P->d_fpv);
  cudaFree(P->d_nfp);
  P->d_fpk = P->d_fpv = nullptr;
  P->d_nfp = nullptr;
  P->fp_cap = 0;
  P->n_fp.clear();
  if (max_tokens == 0) return KV_OK;
  const size_t rows = (size_t)P->cfg.max_requests * P->cfg.num_kv_heads * (size_t)max_tokens;
  const size_t bytes = rows * kHeadDim * sizeof(uint16_t);
  if (cudaMalloc(&P->d_fpk, bytes) != cudaSuccess || cudaMalloc(&P->d_fpv, bytes) != cudaSuccess ||
      cudaMalloc(&P->d_nfp, (size_t)P->cfg.max_requests * sizeof(int32_t)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(P->d_fpk);
    cudaFree(P->d_fpv);
    cudaFree(P->d_nfp);
    P->d_fpk = P->d_fpv = nullptr;
    P->d_nfp = nullptr;
    return fail(KV_ERR_OOM, "kv_fp_configure: cannot allocate 2 x %zu bytes of lists", bytes);
  }
  KV_CUDA(cudaMemset(P->d_nfp, 0, (size_t)P->cfg.max_requests * sizeof(int32_t)));
  KV_CUDA(cudaDeviceSynchronize());
  P->fp_cap = max_tokens;
  P->n_fp.assign((size_t)P->cfg.max_requests, 0);
  return KV_OK;
}

kv_status_t kv_fp_append(kv_pool_t* P, const void* k, const void* v, const int32_t* req_ids, int64_t n_tok,
                         void* stream) {
  if (!P || n_tok < 0 || (n_tok > 0 && (!k || !v || !req_ids)))
    return fail(KV_ERR_INVALID_ARG, "kv_fp_append: bad arguments");
  if (P->fp_cap == 0) return fail(KV_ERR_INVALID_ARG, "kv_fp_append: kv_fp_configure has not been called");
  if (n_tok == 0) return KV_OK;
  if (n_tok > INT32_MAX) return fail(KV_ERR_INVALID_ARG, "kv_fp_append: too many tokens");
  // destination slots: each token goes to the end of its request's lists, in order
  std::vector<int32_t> meta((size_t)n_tok * 2);
  std::vector<int32_t> len_req, len_val;
  std::unordered_map<int32_t, int32_t> grow;
  for (int64_t t = 0; t < n_tok; ++t) {
    const int32_t r = req_ids[t];
    if (!req_ok(P, r)) return fail(KV_ERR_INVALID_ARG, "kv_fp_append: request %d not open", r);
    const int32_t at = P->n_fp[r] + grow[r]++;
    if (at >= P->fp_cap)
      return fail(KV_ERR_OOM, "kv_fp_append: request %d's lists would exceed their capacity %d", r, P->fp_cap);
    meta[(size_t)t] = r;
    meta[(size_t)(n_tok + t)] = at;
  }
  for (const auto& g : grow) {
    len_req.push_back(g.first);
    len_val.push_back(P->n_fp[g.first] + g.second);
  }
  DeviceGuard dg(P->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  kv_status_t st = order_after_previous(P, s);
  if (st != KV_OK) return st;
  Upload u;
  const size_t om = u.add(meta.data(), meta.size() * sizeof(int32_t));
  const size_t olr = u.add(len_req.data(), len_req.size() * sizeof(int32_t));
  const size_t olv = u.add(len_val.data(), len_val.size() * sizeof(int32_t));
  if ((st = upload(P, u, s)) != KV_OK) return st;
  const uint8_t* base = (const uint8_t*)P->upload.ptr;
  const int32_t* d_meta = (const int32_t*)(base + om);
  KV_CUDA(launch_fp_store(P, k, v, n_tok, d_meta, d_meta + n_tok, (const int32_t*)(base + olr),
                          (const int32_t*)(base + olv), (int)len_req.size(), s));
  for (size_t i = 0; i < len_req.size(); ++i) P->n_fp[len_req[i]] = len_val[i];
  return KV_OK;
}

kv_status_t kv_fp_drop(kv_pool_t* P, int32_t r, int64_t first, int64_t n_tok, void* stream) {
  if (!P || !req_ok(P, r)) return fail(KV_ERR_INVALID_ARG, "kv_fp_drop: request %d not open", P ? r : -1);
  const int64_t len = P->n_fp.empty() ? 0 : P->n_fp[r];
  if (first < 0 || n_tok < 0 || first + n_tok > len)
    return fail(KV_ERR_INVALID_ARG, "kv_fp_drop: range [%lld, %lld) outside the list of %lld tokens", (long long)first,
                (long long)(first + n_tok), (long long)len);
  if (n_tok == 0) return KV_OK;
  DeviceGuard dg(P->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  kv_status_t st = order_after_previous(P, s);
  if (st != KV_OK) return st;
  const int64_t tail = len - first - n_tok;
  if ((st = ensure(P->fp_scratch, (size_t)std::max<int64_t>(1, 2 * tail * P->cfg.num_kv_heads * kHeadDim * 2))) != KV_OK)
    return st;
  KV_CUDA(launch_fp_move(P, r, (int32_t)(first + n_tok), (int32_t)first, (int32_t)tail, (int32_t)(len - n_tok), s));
  P->n_fp[r] = (int32_t)(len - n_tok);
  return KV_OK;
}

kv_status_t kv_fp_count(kv_pool_t* P, int32_t r, int64_t* n_tok) {
  if (!P || !req_ok(P, r) || !n_tok) return fail(KV_ERR_INVALID_ARG, "kv_fp_count: bad arguments");
  *n_tok = P->n_fp.empty() ? 0 : P->n_fp[r];
  return KV_OK;
}

kv_status_t kv_export_request(kv_pool_t* P, int32_t r, int32_t* ids, uint8_t* is2, uint8_t* fill, uint32_t* live,
                              uint8_t* kc, uint8_t* vc, uint16_t* km, uint16_t* vm) {
  if (!P || !req_ok(P, r)) return fail(KV_ERR_INVALID_ARG, "kv_export_request: request %d not open", r);
  const bool content = kc || vc || km || vm;
  if (content && !(kc && vc && km && vm)) return fail(KV_ERR_INVALID_ARG, "kv_export_request: pass all four content buffers or none");
  const auto& tb = P->reqs[r].table;
  const int hkv = P->cfg.num_kv_heads;
  for (size_t i = 0; i < tb.size(); ++i) {
    if (ids) ids[i] = tb[i];
    if (is2) is2[i] = is_int2(P, tb[i]) ? 1 : 0;
    if (fill) fill[i] = P->fill[tb[i]];
    if (live) live[i] = P->live[tb[i]];
  }
  if (!content) return KV_OK;
  kv_status_t st = kv_pool_sync(P);
  if (st != KV_OK && st != KV_ERR_RANGE) return st;
  DeviceGuard dg(P->cfg.device);
  std::vector<uint8_t> raw((size_t)hkv * kInt4Block);
  for (size_t i = 0; i < tb.size(); ++i) {
    const int32_t id = tb[i];
    const bool i2 = is_int2(P, id), i3 = is_int3(P, id), f4 = is_fp4(P, id);
    const size_t bs = i2 ? kInt2Block : (i3 ? kInt3Block : (f4 ? kFp4Block : kInt4Block));
    const uint8_t* src =
        i2   ? P->d_pool + (size_t)id * hkv * kInt2Block
        : i3 ? P->d_pool + P->int3_offset + (size_t)(id - first_int3(P)) * hkv * kInt3Block
        : f4 ? P->d_pool + P->fp4_offset + (size_t)(id - first_fp4(P)) * hkv * kFp4Block
             : P->d_pool + P->int4_offset + (size_t)(id - P->cfg.n_int2_pages) * hkv * kInt4Block;
    KV_CUDA(cudaMemcpy(raw.data(), src, bs * hkv, cudaMemcpyDeviceToHost));
    for (int h = 0; h < hkv; ++h) {
      const uint8_t* b = raw.data() + (size_t)h * bs;
      const size_t o = (i * hkv + h);
      uint8_t* kco = kc + o * kPage * kHeadDim;
      uint8_t* vco = vc + o * kPage * kHeadDim;
      uint16_t* kmo = km + o * 256;
      uint16_t* vmo = vm + o * 256;
      auto h16 = [&](int off) { uint16_t x; std::memcpy(&x, b + off, 2); return x; };
      if (f4) {
        // E2M1 codes; scale/zero pairs {s, 0} (symmetric groups)
        for (int t = 0; t < kPage; ++t)
          for (int c = 0; c < kHeadDim; ++c) {
            kco[t * kHeadDim + c] = (b[f4k_byte(t, c)] >> f4k_shift(c)) & 15;
            vco[t * kHeadDim + c] = (b[f4v_byte(t, c)] >> f4v_shift(t)) & 15;
          }
        for (int t = 0; t < kPage; ++t)
          for (int gr = 0; gr < 4; ++gr) {
            kmo[(t * 4 + gr) * 2] = h16(kF4KScale + 8 * t + 2 * gr);
            kmo[(t * 4 + gr) * 2 + 1] = 0;
            vmo[(t * 4 + gr) * 2] = h16(kF4VScale + 2 * v_meta_index(t, gr));
            vmo[(t * 4 + gr) * 2 + 1] = 0;
          }
        continue;
      }
      for (int t = 0; t < kPage; ++t)
        for (int c = 0; c < kHeadDim; ++c) {
          if (i3) {
            kco[t * kHeadDim + c] = (uint8_t)(((b[i3k_lo_byte(t, c)] >> i3k_lo_shift(c)) & 3) |
                                              (((b[i3k_hi_byte(t, c)] >> i3k_hi_shift(c)) & 1) << 2));
            vco[t * kHeadDim + c] = (uint8_t)(((b[i3v_lo_byte(t, c)] >> i3v_lo_shift(t)) & 3) |
                                              (((b[i3v_hi_byte(t, c)] >> i3v_hi_shift(t, c)) & 1) << 2));
            continue;
          }
          kco[t * kHeadDim + c] = i2 ? (b[i2k_byte(t, c)] >> i2k_shift(c)) & 3 : (b[i4k_byte(t, c)] >> i4k_shift(c)) & 15;
          vco[t * kHeadDim + c] = i2 ? (b[i2v_byte(t, c)] >> i2v_shift(t)) & 3 : (b[i4v_byte(t, c)] >> i4v_shift(t)) & 15;
        }
      const int vbase = i2 ? kI2VMeta : (i3 ? kI3VMeta : kI4VMeta);
      const int kbase = i3 ? kI3KMeta : kI4KMeta;
      for (int t = 0; t < kPage; ++t)
        for (int gr = 0; gr < 4; ++gr) {
          vmo[(t * 4 + gr) * 2] = h16(vbase + 2 * v_meta_index(t, gr));
          vmo[(t * 4 + gr) * 2 + 1] = h16(vbase + 256 + 2 * v_meta_index(t, gr));
          if (!i2) {
            kmo[(t * 4 + gr) * 2] = h16(kbase + 16 * t + 4 * gr);
            kmo[(t * 4 + gr) * 2 + 1] = h16(kbase + 16 * t + 4 * gr + 2);
          }
        }
      if (i2)
        for (int c = 0; c < kHeadDim; ++c) {
          kmo[c * 2] = h16(kI2KMeta + 2 * i2k_meta_index(c));
          kmo[c * 2 + 1] = h16(kI2KMeta + 256 + 2 * i2k_meta_index(c));
        }
    }
  }
  return st;
}

}  // extern "C"

namespace {

// Split planner (Tangram, ahead-of-time load balancing: the CTA count comes
// from the occupancy API and work is partitioned before the launch).  All
// (batch row, kv head) units' pages, in order, are cut into n_ctas contiguous
// ranges of about equal cost; a range that crosses unit boundaries becomes one
// split per unit.  A page costs what the chosen scan kernel spends on a page
// of its precision (PageCost), so INT2 and INT4 pages are weighed fairly.

kv_status_t build_plan(kv_pool* P, const int32_t* req_ids, int32_t batch, int32_t hq, int32_t impl,
                       cudaStream_t s) {
  const int hkv = P->cfg.num_kv_heads, g = hq / hkv;
  // A plan stays valid while the batch is the same and no table has shrunk:
  // splits are table index ranges and each unit's last one is open-ended.
  // Tables that grew add their new pages to the tail CTA, so the plan is
  // rebuilt once a table has grown past the slack (or an empty table gained
  // pages, which has no split yet).
  // Full-precision splits follow the same rule: a unit's last one is
  // open-ended, and the plan is rebuilt once a list has grown by 64 tokens, has
  // shrunk, or was empty.
  bool same = P->plan_impl == impl && P->plan_hq == hq && (int32_t)P->plan_req.size() == batch;
  for (int32_t b = 0; same && b < batch; ++b) {
    const int32_t len = (int32_t)P->reqs[req_ids[b]].table.size(), len0 = P->plan_len[b];
    same = P->plan_req[b] == req_ids[b] && len >= len0 && len - len0 <= P->plan_slack && (len0 > 0 || len == 0);
    const int32_t nf = P->n_fp.empty() ? 0 : P->n_fp[req_ids[b]], nf0 = P->plan_nfp[b];
    same = same && nf >= nf0 && nf - nf0 < 2 * kFpMinTokens && (nf0 > 0 || nf == 0);
    // with per-head exclusion, splits may leave out positions found dead: an
    // entry erased or moved (not an append at the end) plans again
    same = same && (P->hdead.empty() || P->plan_ver[b] == P->reqs[req_ids[b]].shape);
  }
  if (same) return KV_OK;

  const bool mma = impl == KV_DECODE_MMA;
  const int per_sm = mma ? decode_mma_workers_per_sm(g) : decode_simt_ctas_per_sm(g);
  HostPlan hp;
  plan_decode(P, req_ids, batch, (int64_t)P->sm_count * per_sm, mma ? kMinPagesPerWarp : kMinPagesPerCta,
              mma ? mma_page_cost(g) : kSimtPageCost, mma, hp);
  Upload up;
  const size_t ou = up.add(hp.units.data(), hp.units.size() * sizeof(Unit));
  const size_t os = up.add(hp.splits.data(), hp.splits.size() * sizeof(Split));
  const size_t oc = up.add(hp.cta_split.data(), hp.cta_split.size() * sizeof(int32_t));
  const size_t of = up.add(hp.fp_wsplit.data(), hp.fp_wsplit.size() * sizeof(int32_t));
  kv_status_t st = ensure(P->plan, up.size);
  if (st != KV_OK) return st;
  if ((st = h2d(P, P->plan.ptr, up, s)) != KV_OK) return st;
  P->plan_units_off = ou;
  P->plan_splits_off = os;
  P->plan_cta_off = oc;
  P->n_units = (int32_t)hp.units.size();
  P->n_splits = (int32_t)hp.splits.size();
  P->n_page_splits = hp.n_page_splits;
  P->plan_fpw_off = of;
  P->n_fpw = (int32_t)hp.fp_wsplit.size() - 1;
  P->n_ctas = (int32_t)hp.n_ctas();
  P->plan_req.assign(req_ids, req_ids + batch);
  P->plan_len.resize(batch);
  P->plan_nfp.resize(batch);
  P->plan_ver.resize(batch);
  for (int32_t b = 0; b < batch; ++b) P->plan_ver[b] = P->reqs[req_ids[b]].shape;
  for (int32_t b = 0; b < batch; ++b) P->plan_nfp[b] = P->n_fp.empty() ? 0 : P->n_fp[req_ids[b]];
  int64_t total_pages = 0;
  for (int32_t b = 0; b < batch; ++b) {
    P->plan_len[b] = (int32_t)P->reqs[req_ids[b]].table.size();
    total_pages += (int64_t)P->plan_len[b] * hkv;
  }
  // growth a tail worker absorbs before the plan is rebuilt: 5% of a worker's share
  P->plan_slack = (int32_t)std::max<int64_t>(1, total_pages / std::max<int64_t>(1, P->n_ctas) / 20);
  P->plan_hq = hq;
  P->plan_impl = impl;
  return KV_OK;
}

}  // namespace

extern "C" {

kv_status_t kv_decode_attn(kv_pool_t* P, const void* q, const int32_t* req_ids, int32_t batch, int32_t hq,
                           float softmax_scale, float* out, void* stream) {
  if (!P) return fail(KV_ERR_INVALID_ARG, "kv_decode_attn: null pool");
  if (!q || !out || !req_ids || batch < 1) return fail(KV_ERR_INVALID_ARG, "kv_decode_attn: null pointer or batch < 1");
  const int hkv = P->cfg.num_kv_heads;
  if (hq < hkv || hq % hkv != 0 || hq / hkv > 8)
    return fail(KV_ERR_INVALID_ARG, "kv_decode_attn: num_q_heads %d must be a multiple of %d with ratio <= 8", hq, hkv);
  if (!std::isfinite(softmax_scale)) return fail(KV_ERR_INVALID_ARG, "kv_decode_attn: softmax_scale must be finite");
  for (int32_t b = 0; b < batch; ++b)
    if (!req_ok(P, req_ids[b])) return fail(KV_ERR_INVALID_ARG, "kv_decode_attn: request %d not open", req_ids[b]);
  const int32_t impl = P->decode_impl == KV_DECODE_AUTO ? KV_DECODE_MMA : P->decode_impl;
  DeviceGuard dg(P->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  kv_status_t st = order_after_previous(P, s);
  if (st != KV_OK) return st;
  if ((st = build_plan(P, req_ids, batch, hq, impl, s)) != KV_OK) return st;
  const int g = hq / hkv;
  if ((st = ensure(P->partials, (size_t)std::max(P->n_splits, 1) * g * (kHeadDim + 4) * sizeof(float))) != KV_OK)
    return st;
  if (impl == KV_DECODE_MMA && (st = ensure(P->frags, (size_t)std::max(P->n_units, 1) * decode_mma_frag_bytes())) != KV_OK)
    return st;
  const uint8_t* base = (const uint8_t*)P->plan.ptr;
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  const Unit* du = (const Unit*)(base + P->plan_units_off);
  const Split* dsp = (const Split*)(base + P->plan_splits_off);
  const int32_t* dct = (const int32_t*)(base + P->plan_cta_off);
  const bool rec = P->timing && (P->timing_seen++ % P->timing_every) == 0;
  cudaEvent_t* tv = rec ? &P->tev[3 * (size_t)(P->timed_calls % kTimingRing)] : nullptr;
  if (tv) KV_CUDA(cudaEventRecord(tv[0], s));
  P->merge_event = tv ? tv[1] : nullptr;
  P->fp_pending = FpLaunch{dsp + P->n_page_splits, (const int32_t*)(base + P->plan_fpw_off), P->n_fpw,
                            P->n_page_splits};
  if (impl == KV_DECODE_MMA)
    KV_CUDA(launch_decode_mma(P, q, hq, scale_log2, du, P->n_units, dsp, dct, P->n_ctas, P->frags.ptr,
                              (float*)P->partials.ptr, out, s));
  else
    KV_CUDA(launch_decode_simt(P, q, hq, scale_log2, du, P->n_units, dsp, dct, P->n_ctas, (float*)P->partials.ptr, out, s));
  if (tv) {
    KV_CUDA(cudaEventRecord(tv[2], s));
    ++P->timed_calls;
  }
  P->merge_event = nullptr;
  P->stat_req.assign(req_ids, req_ids + batch);
  P->stat_hq = hq;
  P->stat_skip_dead = false;
  return KV_OK;
}

kv_status_t kv_decode_timing(kv_pool_t* P, int32_t enable, int64_t* n_calls, float* scan_ms, float* decode_ms) {
  if (!P) return fail(KV_ERR_INVALID_ARG, "kv_decode_timing: null pool");
  DeviceGuard dg(P->cfg.device);
  if (n_calls) *n_calls = P->timed_calls;
  if (scan_ms) *scan_ms = -1.0f;
  if (decode_ms) *decode_ms = -1.0f;
  if (P->timed_calls > 0 && (scan_ms || decode_ms)) {
    const int64_t n = std::min<int64_t>(P->timed_calls, kTimingRing);
    const int64_t last = (P->timed_calls - 1) % kTimingRing;
    KV_CUDA(cudaEventSynchronize(P->tev[3 * (size_t)last + 2]));
    double a = 0.0, b = 0.0;
    for (int64_t k = 0; k < n; ++k) {
      float x = 0.0f, y = 0.0f;
      KV_CUDA(cudaEventElapsedTime(&x, P->tev[3 * (size_t)k], P->tev[3 * (size_t)k + 1]));
      KV_CUDA(cudaEventElapsedTime(&y, P->tev[3 * (size_t)k], P->tev[3 * (size_t)k + 2]));
      a += x;
      b += y;
    }
    if (scan_ms) *scan_ms = (float)(a / (double)n);
    if (decode_ms) *decode_ms = (float)(b / (double)n);
  }
  if (enable < 0) return fail(KV_ERR_INVALID_ARG, "kv_decode_timing: enable must be >= 0");
  if (enable) {
    if (P->tev.empty()) {
      P->tev.assign(3 * (size_t)kTimingRing, nullptr);
      for (auto& e : P->tev) KV_CUDA(cudaEventCreate(&e));
    }
    P->timed_calls = 0;
    P->timing_seen = 0;
    P->timing_every = enable;
  }
  P->timing = enable != 0;
  return KV_OK;
}

kv_status_t kv_pool_launch_count(kv_pool_t* P, int64_t* n) {
  if (!P || !n) return fail(KV_ERR_INVALID_ARG, "kv_pool_launch_count: null argument");
  *n = P->launches;
  return KV_OK;
}

kv_status_t kv_last_decode_stats(kv_pool_t* P, int64_t* kv_bytes, int32_t* n_splits, int64_t* n_pages) {
  if (!P) return fail(KV_ERR_INVALID_ARG, "kv_last_decode_stats: null pool");
  int64_t bytes = 0, pages = 0;
  const int64_t hkv = P->cfg.num_kv_heads;
  for (int32_t r : P->stat_req) {
    if (!req_ok(P, r)) continue;
    for (int32_t id : P->reqs[r].table) {
      // with per-head exclusion (or after a grouped decode), a page with no
      // live slot for a head is not read for it
      int64_t heads = hkv;
      if (!P->hdead.empty())
        for (int h = 0; h < hkv; ++h) heads -= (P->live[id] & ~P->hdead[(size_t)id * hkv + h]) == 0u ? 1 : 0;
      else if (P->stat_skip_dead && P->live[id] == 0u)
        heads = 0;
      // INT4: 160 bytes per written slot (codes 128, scale/zero 32); INT3: 128 (96 + 32); FP4: 144 (128 + 16)
      bytes += is_int2(P, id) ? (int64_t)kInt2Block * heads
                              : (int64_t)P->fill[id] * (is_int3(P, id) ? 128 : (is_fp4(P, id) ? 144 : 160)) * heads;
      bytes += 8;
      ++pages;
    }
    bytes += (int64_t)P->stat_hq * kHeadDim * (2 + 4);
    if (!P->n_fp.empty()) bytes += (int64_t)P->n_fp[r] * hkv * kHeadDim * 2 * 2;   // full-precision K and V
  }
  if (kv_bytes) *kv_bytes = bytes;
  if (n_splits) *n_splits = P->n_splits;
  if (n_pages) *n_pages = pages * hkv;
  return KV_OK;
}

}  // extern "C"

namespace {

// Grouped split planner (Tangram, head groups with their own budgets: every
// group is a pool of its own, and one scan walks them all).  The units of all
// pools in output order: batch row, then kv head across the pools, pool 0's
// kv heads first; a unit's pages are its pool's table for the row's request.
// The cut is plan_decode's: every worker gets about the same cost.  The
// grouped scan skips every page with no live slot for the unit's kv head, so
// a full such page costs nothing, and a unit's leading ones are left out of
// its splits (the plan is rebuilt when a table's entries are erased or
// moved, so those positions keep holding dead pages).
struct GroupHostPlan {
  std::vector<Unit> units;
  std::vector<Split> splits;
  std::vector<int32_t> wsplit;
  int64_t pages = 0;
};

void plan_decode_groups(kv_pool* const* pools, int n_pools, const int32_t* req_ids, int32_t batch, int64_t n_workers,
                        int64_t min_pages, PageCost pc, GroupHostPlan& out) {
  int thkv = 0;
  for (int p = 0; p < n_pools; ++p) thkv += pools[p]->cfg.num_kv_heads;
  const size_t nu = (size_t)batch * thkv;
  std::vector<int32_t> u_pool(nu), u_head(nu), u_req(nu), u_npos(nu), u_lead(nu);
  for (int32_t b = 0; b < batch; ++b) {
    size_t u = (size_t)b * thkv;
    for (int p = 0; p < n_pools; ++p) {
      const kv_pool* P = pools[p];
      const int32_t r = req_ids[(size_t)p * batch + b];
      const auto& tb = P->reqs[r].table;
      int32_t lead = 0;
      for (int32_t id : tb) lead += id < P->cfg.n_int2_pages ? 1 : 0;
      for (int h = 0; h < P->cfg.num_kv_heads; ++h, ++u) {
        u_pool[u] = p;
        u_head[u] = h;
        u_req[u] = r;
        u_npos[u] = (int32_t)tb.size();
        u_lead[u] = lead;
      }
    }
  }
  // per unit: the cost of its first i pages in scan order
  std::vector<int64_t> off(nu + 1, 0);
  for (size_t u = 0; u < nu; ++u) off[u + 1] = off[u] + u_npos[u] + 1;
  std::vector<double> pre((size_t)off[nu]);
  double total = 0.0;
  int64_t pages = 0;
  for (size_t u = 0; u < nu; ++u) {
    const kv_pool* P = pools[u_pool[u]];
    const auto& tb = P->reqs[u_req[u]].table;
    const int hkv = P->cfg.num_kv_heads, h = u_head[u];
    const int64_t n2 = P->cfg.n_int2_pages, n3b = first_int3(P), nfb = first_fp4(P);
    double* pb = &pre[(size_t)off[u]];
    ScanOrder so;
    so.start(0, u_npos[u], u_lead[u]);
    pb[0] = 0.0;
    for (int32_t i = 0; i < u_npos[u]; ++i) {
      const int32_t id = tb[so.next()];
      const uint32_t hd = P->hdead.empty() ? 0u : P->hdead[(size_t)id * hkv + h];
      const bool dead = P->fill[id] == kPage && (P->live[id] & ~hd) == 0u;
      const double c = id < n2 ? pc.int2 : (id >= nfb ? pc.fp4 : (id >= n3b ? pc.int3 : pc.int4));
      pb[i + 1] = pb[i] + (dead ? 0.0 : c);
    }
    total += pb[u_npos[u]];
    pages += u_npos[u];
  }
  out.pages = pages;
  const int64_t n = std::max<int64_t>(1, std::min<int64_t>(n_workers, pages / std::max<int64_t>(1, min_pages)));
  out.units.assign(nu, Unit{});
  out.splits.clear();
  out.wsplit.assign((size_t)n + 1, 0);
  const double scale = total > 0.0 ? (double)n / total : 0.0;
  auto worker = [&](double c) { return std::min<int64_t>(n - 1, (int64_t)(c * scale)); };
  int64_t cur = 0;   // worker receiving the current split
  double U = 0.0;    // cost before the current unit
  for (size_t u = 0; u < nu; ++u) {
    const double* pb = &pre[(size_t)off[u]];
    const int32_t npos = u_npos[u];
    Unit& un = out.units[u];
    un.b = (int32_t)(u / thkv);
    un.req = u_req[u];
    un.kvh = (int32_t)(u % thkv);
    un.pad = u_pool[u];
    un.split_begin = (int32_t)out.splits.size();
    auto split = [&](int32_t b0, int32_t e0) {
      return Split{(int32_t)u, b0, e0, u_req[u], npos, u_lead[u], {u_pool[u], u_head[u]}};
    };
    int32_t i = 0;
    while (i < npos && pb[i + 1] == pb[i]) ++i;
    if (i == npos && npos > 0) {
      // nothing live: one empty split, open-ended so that later pages are scanned
      const int64_t j = worker(U + pb[npos]);
      while (cur < j) out.wsplit[(size_t)++cur] = (int32_t)out.splits.size();
      out.splits.push_back(split(npos, npos));
    }
    while (i < npos) {
      const int64_t j = worker(U + pb[i]);
      while (cur < j) out.wsplit[(size_t)++cur] = (int32_t)out.splits.size();
      int32_t lo = i + 1, hi = npos;
      while (lo < hi) {
        const int32_t mid = lo + (hi - lo) / 2;
        if (worker(U + pb[mid]) > j) hi = mid;
        else lo = mid + 1;
      }
      out.splits.push_back(split(i, lo));
      i = lo;
    }
    U += pb[npos];
    un.n_splits = (int32_t)out.splits.size() - un.split_begin;
    if (un.n_splits > 0) out.splits.back().page_end = -1;   // open-ended: appended pages are scanned
    un.fp_begin = (int32_t)out.splits.size();
    un.n_fp_splits = 0;
  }
  while (cur < n) out.wsplit[(size_t)++cur] = (int32_t)out.splits.size();
}

bool same_pools(const std::vector<GroupPool>& a, const std::vector<GroupPool>& b) {
  return a.size() == b.size() && (a.empty() || std::memcmp(a.data(), b.data(), a.size() * sizeof(GroupPool)) == 0);
}

// The grouped plan and the pools' descriptors, cached in the first pool under
// the rules of build_plan (same pools, rows and requests; no table shrunk,
// erased from or reordered; growth within the slack).
kv_status_t build_group_plan(kv_pool* const* pools, int n_pools, const int32_t* req_ids, int32_t batch, int32_t hq,
                             const std::vector<GroupPool>& gp, cudaStream_t s) {
  kv_pool* P = pools[0];
  const size_t nr = (size_t)n_pools * batch;
  bool same = P->gplan_hq == hq && P->gplan_req.size() == nr && P->gplan_owner.size() == (size_t)n_pools &&
              same_pools(P->gplan_pools, gp);
  for (int p = 0; same && p < n_pools; ++p) same = P->gplan_owner[p] == pools[p]->serial;
  for (size_t k = 0; same && k < nr; ++k) {
    const kv_pool* Q = pools[k / batch];
    const int32_t r = req_ids[k];
    const int32_t len = (int32_t)Q->reqs[r].table.size(), len0 = P->gplan_len[k];
    same = P->gplan_req[k] == r && len >= len0 && len - len0 <= P->gplan_slack && (len0 > 0 || len == 0) &&
           P->gplan_ver[k] == Q->reqs[r].shape;
  }
  if (same) return KV_OK;
  int thkv = 0;
  for (int p = 0; p < n_pools; ++p) thkv += pools[p]->cfg.num_kv_heads;
  const int g = hq / thkv;
  GroupHostPlan hp;
  plan_decode_groups(pools, n_pools, req_ids, batch, (int64_t)P->sm_count * decode_mma_workers_per_sm(g),
                     kMinPagesPerWarp, mma_page_cost(g), hp);
  Upload up;
  const size_t ou = up.add(hp.units.data(), hp.units.size() * sizeof(Unit));
  const size_t os = up.add(hp.splits.data(), hp.splits.size() * sizeof(Split));
  const size_t ow = up.add(hp.wsplit.data(), hp.wsplit.size() * sizeof(int32_t));
  const size_t og = up.add(gp.data(), gp.size() * sizeof(GroupPool));
  kv_status_t st = ensure(P->gplan, up.size);
  if (st != KV_OK) return st;
  if ((st = h2d(P, P->gplan.ptr, up, s)) != KV_OK) return st;
  P->gplan_units_off = ou;
  P->gplan_splits_off = os;
  P->gplan_wsplit_off = ow;
  P->gplan_pools_off = og;
  P->gplan_units = (int32_t)hp.units.size();
  P->gplan_splits = (int32_t)hp.splits.size();
  P->gplan_workers = (int32_t)hp.wsplit.size() - 1;
  P->gplan_pools = gp;
  P->gplan_owner.resize(n_pools);
  for (int p = 0; p < n_pools; ++p) P->gplan_owner[p] = pools[p]->serial;
  P->gplan_req.assign(req_ids, req_ids + nr);
  P->gplan_len.resize(nr);
  P->gplan_ver.resize(nr);
  for (size_t k = 0; k < nr; ++k) {
    const kv_pool* Q = pools[k / batch];
    P->gplan_len[k] = (int32_t)Q->reqs[req_ids[k]].table.size();
    P->gplan_ver[k] = Q->reqs[req_ids[k]].shape;
  }
  // growth a tail worker absorbs before the plan is rebuilt: 5% of a worker's
  // share of the (page, kv head) pairs
  P->gplan_slack = (int32_t)std::max<int64_t>(1, hp.pages / std::max<int64_t>(1, P->gplan_workers) / 20);
  P->gplan_hq = hq;
  return KV_OK;
}

}  // namespace

extern "C" kv_status_t kv_decode_attn_groups(kv_pool_t* const* pools, int32_t n_pools, const void* q,
                                             const int32_t* req_ids, int32_t batch, int32_t hq, float softmax_scale,
                                             float* out, void* stream) {
  if (!pools || n_pools < 1 || n_pools > kMaxGroupPools)
    return fail(KV_ERR_INVALID_ARG, "kv_decode_attn_groups: need 1 to %d pools", kMaxGroupPools);
  if (!q || !out || !req_ids || batch < 1)
    return fail(KV_ERR_INVALID_ARG, "kv_decode_attn_groups: null pointer or batch < 1");
  int thkv = 0;
  for (int p = 0; p < n_pools; ++p) {
    if (!pools[p]) return fail(KV_ERR_INVALID_ARG, "kv_decode_attn_groups: pool %d is null", p);
    for (int o = 0; o < p; ++o)
      if (pools[o] == pools[p]) return fail(KV_ERR_INVALID_ARG, "kv_decode_attn_groups: pool %d is listed twice", p);
    if (pools[p]->cfg.device != pools[0]->cfg.device)
      return fail(KV_ERR_INVALID_ARG, "kv_decode_attn_groups: the pools must be on one device");
    thkv += pools[p]->cfg.num_kv_heads;
  }
  if (hq < thkv || hq % thkv != 0 || hq / thkv > 8)
    return fail(KV_ERR_INVALID_ARG,
                "kv_decode_attn_groups: num_q_heads %d must be a multiple of the pools' %d kv heads with ratio <= 8",
                hq, thkv);
  if (!std::isfinite(softmax_scale))
    return fail(KV_ERR_INVALID_ARG, "kv_decode_attn_groups: softmax_scale must be finite");
  for (int p = 0; p < n_pools; ++p)
    for (int32_t b = 0; b < batch; ++b) {
      const int32_t r = req_ids[(size_t)p * batch + b];
      if (!req_ok(pools[p], r))
        return fail(KV_ERR_INVALID_ARG, "kv_decode_attn_groups: request %d of pool %d not open", r, p);
      if (!pools[p]->n_fp.empty() && pools[p]->n_fp[r] > 0)
        return fail(KV_ERR_INVALID_ARG,
                    "kv_decode_attn_groups: request %d of pool %d holds full-precision tokens (not read here)", r, p);
    }
  kv_pool* P = pools[0];
  DeviceGuard dg(P->cfg.device);
  cudaStream_t s = (cudaStream_t)stream;
  kv_status_t st;
  for (int p = 0; p < n_pools; ++p)
    if ((st = order_after_previous(pools[p], s)) != KV_OK) return st;
  std::vector<GroupPool> gp((size_t)n_pools);
  for (int p = 0; p < n_pools; ++p) {
    const kv_pool* Q = pools[p];
    gp[p] = GroupPool{(const uint8_t*)Q->d_pool, Q->int4_offset, (int64_t)Q->cfg.n_int2_pages,
                      (const Entry*)Q->d_table, (const int32_t*)Q->d_ntab,
                      Q->hdead.empty() ? nullptr : (const uint32_t*)Q->d_hdead, Q->d_status + 1,
                      Q->int3_offset, Q->fp4_offset, first_int3(Q), first_fp4(Q),
                      Q->cfg.num_kv_heads, Q->cfg.max_pages_per_request, n_pools, 0};
  }
  if ((st = build_group_plan(pools, n_pools, req_ids, batch, hq, gp, s)) != KV_OK) return st;
  const int g = hq / thkv;
  if ((st = ensure(P->partials, (size_t)std::max(P->gplan_splits, 1) * g * (kHeadDim + 4) * sizeof(float))) != KV_OK)
    return st;
  if ((st = ensure(P->frags, (size_t)std::max(P->gplan_units, 1) * decode_mma_frag_bytes())) != KV_OK) return st;
  const uint8_t* base = (const uint8_t*)P->gplan.ptr;
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  const bool rec = P->timing && (P->timing_seen++ % P->timing_every) == 0;
  cudaEvent_t* tv = rec ? &P->tev[3 * (size_t)(P->timed_calls % kTimingRing)] : nullptr;
  if (tv) KV_CUDA(cudaEventRecord(tv[0], s));
  P->merge_event = tv ? tv[1] : nullptr;
  P->fp_pending = FpLaunch{};
  bool extra = false;   // some pool holds INT3 or FP4 pages: the scan variant that reads them
  for (int p = 0; p < n_pools; ++p) extra |= pools[p]->cfg.n_int3_pages > 0 || pools[p]->cfg.n_fp4_pages > 0;
  KV_CUDA(launch_decode_mma(P, q, hq, scale_log2, (const Unit*)(base + P->gplan_units_off), P->gplan_units,
                            (const Split*)(base + P->gplan_splits_off), (const int32_t*)(base + P->gplan_wsplit_off),
                            P->gplan_workers, P->frags.ptr, (float*)P->partials.ptr, out, s,
                            (const GroupPool*)(base + P->gplan_pools_off), thkv, extra));
  if (tv) {
    KV_CUDA(cudaEventRecord(tv[2], s));
    ++P->timed_calls;
  }
  P->merge_event = nullptr;
  for (int p = 0; p < n_pools; ++p) {
    pools[p]->stat_req.assign(req_ids + (size_t)p * batch, req_ids + (size_t)(p + 1) * batch);
    pools[p]->stat_hq = pools[p]->cfg.num_kv_heads * g;
    pools[p]->stat_skip_dead = true;
  }
  return KV_OK;
}
