// Full-precision token lists of the decode (HyQuant, Algorithm 3: after the
// quantized prefix the decode scans the vertical-line tokens, the staging
// buffer and the window, all in full precision, under the same online-softmax
// state; Algorithm 4 FREEZE decides which tokens those are).  Each request has
// one list per kv head, K and V in bf16, laid out [request][kv head][slot][128]
// so that a unit's rows are contiguous.
//
// fp_segment_kernel: one warp per split of up to kFpChunk tokens of one unit
// (batch row, kv head).  It writes a partial (acc[128], m, l in the log2
// domain) in the format of the page scans, so the split merge combines both.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kFpWarps = 8;
constexpr int kFpPartStride = kHeadDim + 4;   // the page scans' partial stride

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int G>
__global__ void __launch_bounds__(kFpWarps * 32)
    fp_segment_kernel(const uint16_t* __restrict__ q, int hq, float scale_log2, const Unit* __restrict__ units,
                      const Split* __restrict__ fsplits, int n_fsplits, int first_split,
                      const uint16_t* __restrict__ fpk, const uint16_t* __restrict__ fpv, int fp_cap, int hkv,
                      const int32_t* __restrict__ nfp, float* __restrict__ part) {
  __shared__ __align__(16) float qs[kFpWarps][G][kHeadDim];
  __shared__ float ps[kFpWarps][G][32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sidx = blockIdx.x * kFpWarps + w;
  if (sidx >= n_fsplits) return;   // warps are independent: no block barrier below
  const Split sp = fsplits[sidx];
  const Unit u = units[sp.unit];
  const int n_live = nfp[u.req];
  const int e = sp.page_end < 0 ? n_live : min(sp.page_end, n_live);
  const int a = min(sp.page_begin, e);
  // the unit's q rows, scaled into the log2 domain
  for (int x = lane; x < G * kHeadDim; x += 32) {
    const int h = x / kHeadDim, c = x - h * kHeadDim;
    const uint32_t b = q[((size_t)u.b * hq + (size_t)u.kvh * G + h) * kHeadDim + c];
    qs[w][h][c] = __uint_as_float(b << 16) * scale_log2;
  }
  __syncwarp();
  const size_t row0 = ((size_t)u.req * hkv + u.kvh) * (size_t)fp_cap;
  const uint16_t* K = fpk + row0 * kHeadDim;
  const uint16_t* V = fpv + row0 * kHeadDim;
  float m[G], lsum[G], acc[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    lsum[h] = 0.0f;
    acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.0f;
  }
  for (int t0 = a; t0 < e; t0 += 32) {
    // logits: lane j takes token t0 + j
    const int t = t0 + lane;
    float lg[G];
#pragma unroll
    for (int h = 0; h < G; ++h) lg[h] = 0.0f;
    if (t < e) {
      const uint4* kr = reinterpret_cast<const uint4*>(K + (size_t)t * kHeadDim);
#pragma unroll 4
      for (int x = 0; x < kHeadDim / 8; ++x) {
        const uint4 kk = kr[x];
        const float k0 = bf_lo(kk.x), k1 = bf_hi(kk.x), k2 = bf_lo(kk.y), k3 = bf_hi(kk.y);
        const float k4 = bf_lo(kk.z), k5 = bf_hi(kk.z), k6 = bf_lo(kk.w), k7 = bf_hi(kk.w);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 qa = *reinterpret_cast<const float4*>(&qs[w][h][8 * x]);
          const float4 qb = *reinterpret_cast<const float4*>(&qs[w][h][8 * x + 4]);
          float s = lg[h];
          s = fmaf(k0, qa.x, s);
          s = fmaf(k1, qa.y, s);
          s = fmaf(k2, qa.z, s);
          s = fmaf(k3, qa.w, s);
          s = fmaf(k4, qb.x, s);
          s = fmaf(k5, qb.y, s);
          s = fmaf(k6, qb.z, s);
          s = fmaf(k7, qb.w, s);
          lg[h] = s;
        }
      }
    } else {
#pragma unroll
      for (int h = 0; h < G; ++h) lg[h] = -INFINITY;
    }
    // online softmax: the chunk's maximum per head (warp-uniform), the rescale
    // of what earlier chunks added, this chunk's weights
    float corr[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mx = lg[h];
#pragma unroll
      for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      const float mn = fmaxf(m[h], mx);   // finite: lane 0 holds a token
      corr[h] = m[h] == -INFINITY ? 0.0f : exp2f(m[h] - mn);
      m[h] = mn;
      const float p = t < e ? exp2f(lg[h] - mn) : 0.0f;
      lsum[h] = fmaf(lsum[h], corr[h], p);   // per-lane sums, rescaled alike
      ps[w][h][lane] = p;
    }
    __syncwarp();
    // P.V: lane owns channels 4 lane .. 4 lane + 3
#pragma unroll
    for (int h = 0; h < G; ++h) {
      acc[h][0] *= corr[h];
      acc[h][1] *= corr[h];
      acc[h][2] *= corr[h];
      acc[h][3] *= corr[h];
    }
    const int nt = min(32, e - t0);
    const uint16_t* vr = V + (size_t)t0 * kHeadDim + 4 * lane;
#pragma unroll 4
    for (int j = 0; j < nt; ++j) {
      const uint2 vv = *reinterpret_cast<const uint2*>(vr + (size_t)j * kHeadDim);
      const float v0 = bf_lo(vv.x), v1 = bf_hi(vv.x), v2 = bf_lo(vv.y), v3 = bf_hi(vv.y);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float p = ps[w][h][j];
        acc[h][0] = fmaf(p, v0, acc[h][0]);
        acc[h][1] = fmaf(p, v1, acc[h][1]);
        acc[h][2] = fmaf(p, v2, acc[h][2]);
        acc[h][3] = fmaf(p, v3, acc[h][3]);
      }
    }
    __syncwarp();   // ps is rewritten by the next chunk
  }
  float* out = part + (size_t)(first_split + sidx) * G * kFpPartStride;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float l = lsum[h];
#pragma unroll
    for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
    *reinterpret_cast<float4*>(out + h * kFpPartStride + 4 * lane) =
        make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
    if (lane == 0) {
      out[h * kFpPartStride + kHeadDim] = m[h];
      out[h * kFpPartStride + kHeadDim + 1] = l;
    }
  }
}

// Rows src [n][hkv][128] -> list rows at..at+n of every head of request req;
// then the list length.  V = 8: 16-byte pieces (both sides 16-byte aligned),
// V = 1: single elements.
template <int V>
__global__ void fp_store_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                uint16_t* __restrict__ fpk, uint16_t* __restrict__ fpv, int32_t* __restrict__ nfp,
                                int req, int hkv, int fp_cap, int at, int64_t n) {
  constexpr int kPer = kHeadDim / V;   // pieces per row
  const int64_t total = n * hkv * kPer;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total; x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = x / kPer;   // (token, head) in the source order
    const int piece = (int)(x - row * kPer);
    const int64_t t = row / hkv;
    const int h = (int)(row - t * hkv);
    const size_t dst = ((((size_t)req * hkv + h) * fp_cap) + (size_t)(at + t)) * kHeadDim + (size_t)piece * V;
    const size_t src = (size_t)row * kHeadDim + (size_t)piece * V;
    if constexpr (V == 8) {
      *reinterpret_cast<uint4*>(fpk + dst) = *reinterpret_cast<const uint4*>(k + src);
      *reinterpret_cast<uint4*>(fpv + dst) = *reinterpret_cast<const uint4*>(v + src);
    } else {
      fpk[dst] = k[src];
      fpv[dst] = v[src];
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) nfp[req] = at + (int32_t)n;
}

// Rows [at, at + n) of every head of request req, to or from a scratch
// buffer [2][hkv][n][128] (dir 0: list -> scratch, dir 1: scratch -> list;
// the second call also sets the list length).
__global__ void fp_move_kernel(uint16_t* __restrict__ fpk, uint16_t* __restrict__ fpv, uint4* __restrict__ scratch,
                               int32_t* __restrict__ nfp, int req, int hkv, int fp_cap, int at, int n, int dir,
                               int new_len) {
  constexpr int kPer = kHeadDim / 8;
  const int64_t per_list = (int64_t)hkv * n * kPer;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < 2 * per_list;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int which = x >= per_list;
    const int64_t y = x - which * per_list;
    const int64_t row = y / kPer;   // (head, token) in scratch order
    const int piece = (int)(y - row * kPer);
    const int h = (int)(row / n), t = (int)(row - (int64_t)h * n);
    uint4* list = reinterpret_cast<uint4*>(which ? fpv : fpk) +
                  ((((size_t)req * hkv + h) * fp_cap) + (size_t)(at + t)) * kPer + piece;
    if (dir == 0) scratch[x] = *list;
    else *list = scratch[x];
  }
  if (dir == 1 && blockIdx.x == 0 && threadIdx.x == 0) nfp[req] = new_len;
}

int grid_for(int64_t work, int sm_count) {
  const int64_t g = (work + 255) / 256;
  return (int)std::max<int64_t>(1, std::min<int64_t>(g, (int64_t)sm_count * 8));
}

}  // namespace

cudaError_t launch_fp_segments(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units,
                               const Split* d_fsplits, int n_fsplits, int first_split, float* d_part, cudaStream_t s) {
  if (n_fsplits <= 0) return cudaSuccess;
  const int hkv = P->cfg.num_kv_heads;
  const dim3 grid((unsigned)((n_fsplits + kFpWarps - 1) / kFpWarps)), block(kFpWarps * 32);
  const uint16_t* qq = (const uint16_t*)q;
#define KVQ_FP_CASE(g)                                                                                        \
  case g:                                                                                                     \
    fp_segment_kernel<g><<<grid, block, 0, s>>>(qq, hq, scale_log2, d_units, d_fsplits, n_fsplits, first_split, \
                                                P->d_fpk, P->d_fpv, P->fp_cap, hkv, P->d_nfp, d_part);        \
    break;
  switch (hq / hkv) {
    KVQ_FP_CASE(1)
    KVQ_FP_CASE(2)
    KVQ_FP_CASE(3)
    KVQ_FP_CASE(4)
    KVQ_FP_CASE(5)
    KVQ_FP_CASE(6)
    KVQ_FP_CASE(7)
    KVQ_FP_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef KVQ_FP_CASE
  ++P->launches;
  return cudaGetLastError();
}

cudaError_t launch_fp_store(kv_pool* P, int32_t req, const void* k, const void* v, int64_t n, int32_t at,
                            cudaStream_t s) {
  const int hkv = P->cfg.num_kv_heads;
  const bool wide = ((uintptr_t)k % 16 == 0) && ((uintptr_t)v % 16 == 0);
  const int64_t work = n * hkv * (wide ? kHeadDim / 8 : kHeadDim);
  const int grid = grid_for(work, P->sm_count);
  if (wide)
    fp_store_kernel<8><<<grid, 256, 0, s>>>((const uint16_t*)k, (const uint16_t*)v, P->d_fpk, P->d_fpv, P->d_nfp, req,
                                            hkv, P->fp_cap, at, n);
  else
    fp_store_kernel<1><<<grid, 256, 0, s>>>((const uint16_t*)k, (const uint16_t*)v, P->d_fpk, P->d_fpv, P->d_nfp, req,
                                            hkv, P->fp_cap, at, n);
  ++P->launches;
  return cudaGetLastError();
}

cudaError_t launch_fp_move(kv_pool* P, int32_t req, int32_t from, int32_t to, int32_t n, int32_t new_len,
                           cudaStream_t s) {
  const int hkv = P->cfg.num_kv_heads;
  const int64_t work = 2 * (int64_t)hkv * n * (kHeadDim / 8);
  const int grid = grid_for(work, P->sm_count);
  uint4* scratch = (uint4*)P->fp_scratch.ptr;
  fp_move_kernel<<<grid, 256, 0, s>>>(P->d_fpk, P->d_fpv, scratch, P->d_nfp, req, hkv, P->fp_cap, from, n, 0, new_len);
  fp_move_kernel<<<grid, 256, 0, s>>>(P->d_fpk, P->d_fpv, scratch, P->d_nfp, req, hkv, P->fp_cap, to, n, 1, new_len);
  P->launches += 2;
  return cudaGetLastError();
}

}  // namespace kvq
