// kv_decode_attn_noalloc: the decode of kv_decode_attn without any device
// allocation.  kv_decode_attn keeps its split plan and split partials in
// pool-owned buffers that grow with cudaMalloc when a bigger batch arrives;
// this entry point puts both in one fixed, file-scope device array instead,
// for callers that cannot allocate device memory at decode time.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "kvq_internal.h"

namespace kvq {
namespace {

// Scratch for one call: the units of the plan, the per-unit q operands of the
// tensor-core scan, the splits, then the split partials (g x 132 floats per
// split).  Every GPU that loads the library
// holds this array until the process exits.  Nothing in it has to start at
// zero: the plan is copied in by each call and every partial the merge reads
// is written by the scan kernel of the same call.  Calls whose device work
// overlaps (different streams, or another pool) race on it.
constexpr size_t kScratchBytes = size_t(64) << 20;
constexpr int kMaxUnits = 4096;
__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

kv_status_t nfail(kv_status_t st, const char* msg) {
  set_last_error(msg);
  return st;
}

// Device address of the array for `device` (which must be current).  The
// first call per device resolves it; later calls reuse the cached pointer.
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" kv_status_t kv_decode_attn_noalloc(kv_pool_t* P, const void* q, const int32_t* req_ids, int32_t batch,
                                              int32_t hq, float softmax_scale, float* out, void* stream) {
  if (!P || !q || !out || !req_ids || batch < 1)
    return nfail(KV_ERR_INVALID_ARG, "kv_decode_attn_noalloc: null pointer or batch < 1");
  const int hkv = P->cfg.num_kv_heads;
  if (hq < hkv || hq % hkv != 0 || hq / hkv > 8)
    return nfail(KV_ERR_INVALID_ARG, "kv_decode_attn_noalloc: num_q_heads must be a multiple of num_kv_heads, ratio <= 8");
  if (!std::isfinite(softmax_scale)) return nfail(KV_ERR_INVALID_ARG, "kv_decode_attn_noalloc: softmax_scale must be finite");
  for (int32_t b = 0; b < batch; ++b)
    if (req_ids[b] < 0 || req_ids[b] >= P->cfg.max_requests || !P->reqs[req_ids[b]].open)
      return nfail(KV_ERR_INVALID_ARG, "kv_decode_attn_noalloc: a request id is not open");
  const int g = hq / hkv;
  const int64_t n_units = (int64_t)batch * hkv;
  if (n_units > kMaxUnits)
    return nfail(KV_ERR_INVALID_ARG, "kv_decode_attn_noalloc: batch x num_kv_heads exceeds the 4096-unit limit of the fixed scratch");

  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
  if (prev != P->cfg.device && cudaSetDevice(P->cfg.device) != cudaSuccess)
    return nfail(KV_ERR_CUDA, "kv_decode_attn_noalloc: cannot make the pool's device current");
  struct Restore {
    int dev;
    ~Restore() { if (dev >= 0) cudaSetDevice(dev); }
  } restore{prev != P->cfg.device ? prev : -1};

  void* scratch = nullptr;
  if (scratch_address(P->cfg.device, &scratch) != cudaSuccess)
    return nfail(KV_ERR_CUDA, "kv_decode_attn_noalloc: cudaGetSymbolAddress of the scratch array failed");

  // Plan: the same balanced plan as kv_decode_attn, with the worker count
  // capped so that plan + partials fit the scratch (a plan of n workers has
  // at most n + units - 1 page splits, plus the full-precision splits).
  const int32_t impl = P->decode_impl == KV_DECODE_AUTO ? KV_DECODE_MMA : P->decode_impl;
  const bool mma = impl == KV_DECODE_MMA;
  const int per_sm = mma ? decode_mma_workers_per_sm(g) : decode_simt_ctas_per_sm(g);
  const size_t part_bytes = (size_t)g * (kHeadDim + 4) * sizeof(float);
  const size_t units_bytes = align256((size_t)n_units * sizeof(Unit));
  const size_t frags_bytes = mma ? align256((size_t)n_units * decode_mma_frag_bytes()) : 0;
  const int64_t budget = (int64_t)((kScratchBytes - units_bytes - frags_bytes - 1024) /
                                   (sizeof(Split) + sizeof(int32_t) + part_bytes));
  // full-precision splits: at most one per full-precision worker plus one per unit
  const int64_t n_fsplits = P->n_fp.empty() ? 0 : (int64_t)fp_workers(P) + n_units;
  const int64_t n_workers = std::min<int64_t>((int64_t)P->sm_count * per_sm, budget - n_units - 2 * n_fsplits);
  if (n_workers < 1)
    return nfail(KV_ERR_INVALID_ARG, "kv_decode_attn_noalloc: the plan does not fit the fixed scratch");
  HostPlan hp;
  plan_decode(P, req_ids, batch, n_workers, mma ? kMinPagesPerWarp : kMinPagesPerCta,
              mma ? mma_page_cost(g) : kSimtPageCost, mma, hp);
  // layout: units, splits, worker split ranges (the uploaded part), then the
  // per-unit q operands and the partials (written on the device)
  const size_t splits_off = units_bytes;
  const size_t cta_off = align256(splits_off + hp.splits.size() * sizeof(Split));
  const size_t fpw_off = align256(cta_off + hp.cta_split.size() * sizeof(int32_t));
  const size_t frags_off = align256(fpw_off + hp.fp_wsplit.size() * sizeof(int32_t));
  const size_t part_off = frags_off + frags_bytes;
  if (part_off + hp.splits.size() * part_bytes > kScratchBytes)
    return nfail(KV_ERR_INVALID_ARG, "kv_decode_attn_noalloc: the plan does not fit the fixed scratch");
  std::vector<uint8_t> host(frags_off, 0);
  std::memcpy(host.data(), hp.units.data(), hp.units.size() * sizeof(Unit));
  if (!hp.splits.empty()) std::memcpy(host.data() + splits_off, hp.splits.data(), hp.splits.size() * sizeof(Split));
  std::memcpy(host.data() + cta_off, hp.cta_split.data(), hp.cta_split.size() * sizeof(int32_t));
  if (!hp.fp_wsplit.empty())
    std::memcpy(host.data() + fpw_off, hp.fp_wsplit.data(), hp.fp_wsplit.size() * sizeof(int32_t));
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* base = (uint8_t*)scratch;
  if (cudaMemcpyAsync(base, host.data(), frags_off, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return nfail(KV_ERR_CUDA, "kv_decode_attn_noalloc: plan upload failed");
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  const int n_fpw = (int)hp.fp_wsplit.size() - 1;
  P->fp_pending = FpLaunch{(const Split*)(base + splits_off) + hp.n_page_splits, (const int32_t*)(base + fpw_off),
                           n_fpw, hp.n_page_splits};
  const cudaError_t e =
      impl == KV_DECODE_MMA
          ? launch_decode_mma(P, q, hq, scale_log2, (const Unit*)base, (int)n_units, (const Split*)(base + splits_off),
                              (const int32_t*)(base + cta_off), (int)hp.n_ctas(), base + frags_off,
                              (float*)(base + part_off), out, s)
          : launch_decode_simt(P, q, hq, scale_log2, (const Unit*)base, (int)n_units, (const Split*)(base + splits_off),
                               (const int32_t*)(base + cta_off), (int)hp.n_ctas(), (float*)(base + part_off), out, s);
  if (e != cudaSuccess) return nfail(KV_ERR_CUDA, cudaGetErrorString(e));
  return KV_OK;
}
