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

// Scratch for one call: the units and splits of the plan, then the split
// partials (g x 132 floats per split).  Every GPU that loads the library
// holds this array until the process exits.  Nothing in it has to start at
// zero: the plan is copied in by each call and every partial the merge reads
// is written by the scan kernel of the same call.  Calls whose device work
// overlaps (different streams, or another pool) race on it.
constexpr size_t kScratchBytes = size_t(8) << 20;
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

  // Plan: same policy as kv_decode_attn (pure-precision runs cut into
  // near-equal page ranges of about total / (SMs x CTAs per SM) bytes), with
  // the split count capped so plan + partials fit the scratch.
  const int32_t impl = P->decode_impl == KV_DECODE_AUTO ? KV_DECODE_MMA : P->decode_impl;
  const int ctas = impl == KV_DECODE_MMA ? decode_mma_ctas_per_sm(g) : decode_simt_ctas_per_sm(g);
  const size_t part_bytes = (size_t)g * (kHeadDim + 4) * sizeof(float);
  const size_t units_bytes = align256((size_t)n_units * sizeof(Unit));
  const int64_t max_splits = (int64_t)((kScratchBytes - units_bytes - 512) / (sizeof(Split) + part_bytes));
  struct Run { int32_t b, begin, end; bool i2; };
  std::vector<Run> runs;
  double total = 0.0;
  for (int32_t b = 0; b < batch; ++b) {
    const auto& tb = P->reqs[req_ids[b]].table;
    for (int32_t i = 0; i < (int32_t)tb.size();) {
      const bool i2 = tb[i] < P->cfg.n_int2_pages;
      int32_t j = i + 1;
      while (j < (int32_t)tb.size() && (tb[j] < P->cfg.n_int2_pages) == i2) ++j;
      runs.push_back(Run{b, i, j, i2});
      total += (double)(j - i) * (i2 ? kInt2Block : kInt4Block) * hkv;
      i = j;
    }
  }
  const int64_t min_splits = (int64_t)runs.size() * hkv;
  if (min_splits > max_splits)
    return nfail(KV_ERR_INVALID_ARG, "kv_decode_attn_noalloc: the tables hold more precision runs than the fixed scratch can plan");
  const double target = std::min<double>((double)P->sm_count * ctas, (double)(max_splits - min_splits) + 1.0);
  const double chunk = std::max(total / std::max(target, 1.0), 8.0 * kInt2Block);

  std::vector<Unit> units((size_t)n_units);
  std::vector<Split> splits;
  size_t ri = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const size_t r0 = ri;
    while (ri < runs.size() && runs[ri].b == b) ++ri;
    for (int h = 0; h < hkv; ++h) {
      Unit& u = units[(size_t)b * hkv + h];
      u = Unit{};
      u.b = b;
      u.req = req_ids[b];
      u.kvh = h;
      u.split_begin = (int32_t)splits.size();
      for (size_t k = r0; k < ri; ++k) {
        const int32_t np = runs[k].end - runs[k].begin;
        const double bytes = (double)np * (runs[k].i2 ? kInt2Block : kInt4Block);
        const int32_t ns = std::max<int32_t>(1, std::min<int32_t>(np, (int32_t)std::ceil(bytes / chunk)));
        for (int32_t s = 0; s < ns; ++s)
          splits.push_back(Split{(int32_t)((size_t)b * hkv + h), runs[k].begin + (int32_t)((int64_t)np * s / ns),
                                 runs[k].begin + (int32_t)((int64_t)np * (s + 1) / ns), runs[k].i2 ? 1 : 0});
      }
      u.n_splits = (int32_t)splits.size() - u.split_begin;
    }
  }
  if ((int64_t)splits.size() > max_splits)
    return nfail(KV_ERR_INVALID_ARG, "kv_decode_attn_noalloc: the plan does not fit the fixed scratch");

  const size_t splits_off = units_bytes;
  const size_t part_off = align256(splits_off + splits.size() * sizeof(Split));
  std::vector<uint8_t> host(part_off, 0);
  std::memcpy(host.data(), units.data(), units.size() * sizeof(Unit));
  if (!splits.empty()) std::memcpy(host.data() + splits_off, splits.data(), splits.size() * sizeof(Split));
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* base = (uint8_t*)scratch;
  if (cudaMemcpyAsync(base, host.data(), part_off, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return nfail(KV_ERR_CUDA, "kv_decode_attn_noalloc: plan upload failed");
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  const cudaError_t e =
      impl == KV_DECODE_MMA
          ? launch_decode_mma(P, q, hq, scale_log2, (const Unit*)base, (int)n_units, (const Split*)(base + splits_off),
                              (int)splits.size(), (float*)(base + part_off), out, s)
          : launch_decode_simt(P, q, hq, scale_log2, (const Unit*)base, (int)n_units, (const Split*)(base + splits_off),
                               (int)splits.size(), (float*)(base + part_off), out, s);
  if (e != cudaSuccess) return nfail(KV_ERR_CUDA, cudaGetErrorString(e));
  return KV_OK;
}
