// CUDA-core decode kernel (reference / ablation path) and the split merge.
//
// Each CTA scans one split (a run of pages of one (batch row, kv head) unit,
// all of one precision after the INT2-first reorder -- TriAxialKV key design
// 4).  A warp takes one page at a time: it copies the page block to shared
// memory, dequantizes K with fmaf(code, scale, zero) and forms the logits of
// the g packed query heads (HyQuant Algorithm 3, GQA packing), updates the
// online softmax state (m, l, acc) and accumulates P.V with dequantized V.
// Dead slots (evicted or never written) take the sentinel logit -1e4 and V = 0
// (IntentKV, sentinel dead slot).  The warps of a CTA are merged in shared
// memory and the split's (m, l, acc) is written; a second kernel merges splits
// with log-sum-exp (HyQuant ReduceSoftmax; TriAxialKV global LSE reduce).
// Softmax runs in base 2: logits are pre-multiplied by log2(e).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kPartStride = kHeadDim + 4;   // acc[128], m, l, 2 pad: rows stay 16-byte aligned
constexpr float kDeadLogit2 = -1.0e4f * 1.4426950408889634f;   // -1e4 in base-2 units

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}
__device__ __forceinline__ float ld_half(const uint8_t* p) {
  return __half2float(*reinterpret_cast<const __half*>(p));
}

template <int G>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(
    const uint8_t* __restrict__ pool, size_t int4_off, int64_t n2, int hkv, int max_pages,
    const Entry* __restrict__ table, const __nv_bfloat16* __restrict__ q, int hq, float scale_log2,
    const Unit* __restrict__ units, const Split* __restrict__ splits, const int32_t* __restrict__ cta_split,
    const int32_t* __restrict__ ntab, const uint32_t* __restrict__ hdead, float* __restrict__ part, size_t int3_off,
    int64_t n3b, size_t fp4_off, int64_t nfb) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the appends before this decode are done
  asm volatile("griddepcontrol.launch_dependents;");   // the merge may be scheduled as CTAs retire
  __shared__ float qs[G][kHeadDim];
  __shared__ __align__(16) uint8_t buf[kWarps][kInt4Block];
  __shared__ float pb[kWarps][kPage][G];
  __shared__ float wm[kWarps][G], wl[kWarps][G];

  for (int sg = cta_split[blockIdx.x]; sg < cta_split[blockIdx.x + 1]; ++sg) {
  __syncthreads();
  const Split sp = splits[sg];
  const Unit u = units[sp.unit];
  const int page_end = sp.page_end >= 0 ? sp.page_end : ntab[u.req];
  for (int i = threadIdx.x; i < G * kHeadDim; i += kThreads) {
    const int h = i / kHeadDim, c = i % kHeadDim;
    qs[h][c] = __bfloat162float(q[((size_t)u.b * hq + (size_t)u.kvh * G + h) * kHeadDim + c]);
  }
  __syncthreads();

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m[G], l[G], acc[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int a = 0; a < 4; ++a) acc[h][a] = 0.0f;
  }
  const Entry* tab = table + (size_t)u.req * max_pages;
  uint8_t* bw = buf[w];
  for (int pi = sp.page_begin + w; pi < page_end; pi += kWarps) {
    const Entry e = tab[pi];
    // slots excluded for this kv head only read as dead slots too
    const uint32_t live = hdead ? e.live & ~hdead[(size_t)e.id * hkv + u.kvh] : e.live;
    // INT3 ids follow the INT4 ids, FP4 ids the INT3 ids
    const bool i2 = e.id < n2, f4 = e.id >= nfb, i3 = e.id >= n3b && !f4;
    const uint8_t* blk = i2   ? pool + ((size_t)e.id * hkv + u.kvh) * kInt2Block
                         : i3 ? pool + int3_off + ((size_t)(e.id - n3b) * hkv + u.kvh) * kInt3Block
                         : f4 ? pool + fp4_off + ((size_t)(e.id - nfb) * hkv + u.kvh) * kFp4Block
                              : pool + int4_off + ((size_t)(e.id - n2) * hkv + u.kvh) * kInt4Block;
    const int nbytes = i2 ? kInt2Block : (i3 ? kInt3Block : (f4 ? kFp4Block : kInt4Block));
    for (int o = lane * 16; o < nbytes; o += 512)
      *reinterpret_cast<uint4*>(bw + o) = *reinterpret_cast<const uint4*>(blk + o);
    __syncwarp();

    // ---- logits: lane = slot
    const int t = lane;
    float s[G];
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = 0.0f;
    if (i2) {
      for (int c = 0; c < kHeadDim; ++c) {
        const uint32_t code = (bw[i2k_byte(t, c)] >> i2k_shift(c)) & 3u;
        const int mi = i2k_meta_index(c);
        const float kh = __fmaf_rn((float)code, ld_half(bw + kI2KMeta + 2 * mi), ld_half(bw + kI2KMeta + 256 + 2 * mi));
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] = __fmaf_rn(qs[h][c], kh, s[h]);
      }
    } else if (f4) {
      for (int gr = 0; gr < 4; ++gr) {
        const float sf = ld_half(bw + kF4KScale + 8 * t + 2 * gr);
        for (int cc = 0; cc < kGroup; ++cc) {
          const int c = kGroup * gr + cc;
          const float kh = e2m1_value(((uint32_t)bw[f4k_byte(t, c)] >> f4k_shift(c)) & 15u) * sf;
#pragma unroll
          for (int h = 0; h < G; ++h) s[h] = __fmaf_rn(qs[h][c], kh, s[h]);
        }
      }
    } else {
      const int kmeta = i3 ? kI3KMeta : kI4KMeta;
      for (int gr = 0; gr < 4; ++gr) {
        const float sf = ld_half(bw + kmeta + 16 * t + 4 * gr);
        const float zf = ld_half(bw + kmeta + 16 * t + 4 * gr + 2);
        for (int cc = 0; cc < kGroup; ++cc) {
          const int c = kGroup * gr + cc;
          const uint32_t code = i3 ? (((uint32_t)bw[i3k_lo_byte(t, c)] >> i3k_lo_shift(c)) & 3u) |
                                         ((((uint32_t)bw[i3k_hi_byte(t, c)] >> i3k_hi_shift(c)) & 1u) << 2)
                                   : (bw[i4k_byte(t, c)] >> i4k_shift(c)) & 15u;
          const float kh = __fmaf_rn((float)code, sf, zf);
#pragma unroll
          for (int h = 0; h < G; ++h) s[h] = __fmaf_rn(qs[h][c], kh, s[h]);
        }
      }
    }
    const bool alive = (live >> t) & 1u;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float lg = alive ? s[h] * scale_log2 : kDeadLogit2;
      const float mnew = fmaxf(m[h], warp_max(lg));
      const float corr = exp2f(m[h] - mnew);
      const float p = exp2f(lg - mnew);
      l[h] = l[h] * corr + warp_sum(p);
      m[h] = mnew;
      pb[w][t][h] = alive ? p : 0.0f;
#pragma unroll
      for (int a = 0; a < 4; ++a) acc[h][a] *= corr;
    }
    __syncwarp();

    // ---- P.V: lane owns channels 4*lane .. 4*lane+3 (one group)
    const int gr = lane >> 3;
    const int vmeta = i2 ? kI2VMeta : (i3 ? kI3VMeta : (f4 ? kF4VScale : kI4VMeta));
    for (int t2 = 0; t2 < kPage; ++t2) {
      const int mi = v_meta_index(t2, gr);
      const float sf = ld_half(bw + vmeta + 2 * mi), zf = f4 ? 0.0f : ld_half(bw + vmeta + 256 + 2 * mi);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int c = 4 * lane + a;
        const uint32_t code = i2   ? (bw[i2v_byte(t2, c)] >> i2v_shift(t2)) & 3u
                              : i3 ? (((uint32_t)bw[i3v_lo_byte(t2, c)] >> i3v_lo_shift(t2)) & 3u) |
                                         ((((uint32_t)bw[i3v_hi_byte(t2, c)] >> i3v_hi_shift(t2, c)) & 1u) << 2)
                              : f4 ? ((uint32_t)bw[f4v_byte(t2, c)] >> f4v_shift(t2)) & 15u
                                   : (bw[i4v_byte(t2, c)] >> i4v_shift(t2)) & 15u;
        const float vh = f4 ? e2m1_value(code) * sf : __fmaf_rn((float)code, sf, zf);
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h][a] = __fmaf_rn(pb[w][t2][h], vh, acc[h][a]);
      }
    }
    __syncwarp();
  }

  // ---- merge the warps of this CTA
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) { wm[w][h] = m[h]; wl[w][h] = l[h]; }
  }
  __syncthreads();
  float* ab = reinterpret_cast<float*>(&buf[0][0]);   // [kWarps][G][128]
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int a = 0; a < 4; ++a) ab[(w * G + h) * kHeadDim + 4 * lane + a] = acc[h][a];
  __syncthreads();
  float* out = part + (size_t)sg * G * kPartStride;
  const int c = threadIdx.x;
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, wm[ww][h]);
    float L = 0.0f, A = 0.0f;
    for (int ww = 0; ww < kWarps; ++ww) {
      if (wm[ww][h] == -INFINITY) continue;
      const float f = exp2f(wm[ww][h] - M);
      L += wl[ww][h] * f;
      A += ab[(ww * G + h) * kHeadDim + c] * f;
    }
    out[h * kPartStride + c] = A;
    if (c == 0) {
      out[h * kPartStride + kHeadDim] = M;
      out[h * kPartStride + kHeadDim + 1] = L;
    }
  }
  }
}

// One CTA of 8 warps per (unit, head): O = sum_s acc_s 2^(m_s - M) / sum_s
// l_s 2^(m_s - M).  Warp w takes splits w, w + 8, ...: its lanes read those
// splits' m and l at once (lane j: the j-th), the warp takes their maximum
// M_w and weights f = 2^(m - M_w), then every lane adds its four channels of
// each split with the weight fetched by shuffle.  The eight warps' (M_w, L_w,
// A_w) are combined in shared memory.  A unit may have tens of splits (one
// per warp of the tensor-core scan that touched it); this order keeps the
// dependent load rounds at two.
template <int G>
__global__ void __launch_bounds__(256) merge_kernel(const Unit* __restrict__ units, const float* __restrict__ part,
                                                    int hq, float* __restrict__ out) {
  constexpr int kW = 8;
  __shared__ float mpart[kW], lpart[kW];
  __shared__ float4 apart[kW][32];
  const int ui = blockIdx.x / G, h = blockIdx.x - ui * G;
  const Unit u = units[ui];   // the plan is copied in before the launch (not by a kernel): read it first
  // Launched as a programmatic dependent of the scan: wait until the scan grid
  // has completed and its partials are visible (immediate for a plain launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");   // the next call's kernels may be staged
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const size_t rs = (size_t)G * kPartStride;          // stride between splits
  // the unit's page splits, then its full-precision splits
  const float* base = part + ((size_t)u.split_begin * G + h) * kPartStride;
  const float* fbase = part + ((size_t)u.fp_begin * G + h) * kPartStride;
  const int nq = u.n_splits, n = nq + u.n_fp_splits;
  auto split_at = [&](int s) { return s < nq ? base + (size_t)s * rs : fbase + (size_t)(s - nq) * rs; };
  float Mw = -INFINITY, Lw = 0.0f;
  float4 A = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  constexpr int kOne = 12;  // splits per warp read in one round (units of up to kW * kOne splits)
  if (n <= kW * kOne) {
    // every load of the warp's splits at once, then the weights
    const int mine = n > w ? (n - w + kW - 1) / kW : 0;
    float m[kOne], l[kOne];
    float4 a[kOne];
#pragma unroll
    for (int j = 0; j < kOne; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.0f;
      a[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (j < mine) {
        const float* ps = split_at(w + kW * j);
        m[j] = ps[kHeadDim];
        l[j] = ps[kHeadDim + 1];
        a[j] = *reinterpret_cast<const float4*>(ps + 4 * lane);
      }
    }
#pragma unroll
    for (int j = 0; j < kOne; ++j) Mw = fmaxf(Mw, m[j]);
#pragma unroll
    for (int j = 0; j < kOne; ++j) {
      const float f = m[j] == -INFINITY ? 0.0f : exp2f(m[j] - Mw);   // an empty split adds nothing
      Lw = fmaf(f, l[j], Lw);
      A.x = fmaf(a[j].x, f, A.x);
      A.y = fmaf(a[j].y, f, A.y);
      A.z = fmaf(a[j].z, f, A.z);
      A.w = fmaf(a[j].w, f, A.w);
    }
  } else
  for (int s0 = w; s0 < n; s0 += kW * 32) {           // 32 of the warp's splits per round
    const int s = s0 + kW * lane;
    float m = -INFINITY, l = 0.0f;
    if (s < n) {
      m = split_at(s)[kHeadDim];
      l = split_at(s)[kHeadDim + 1];
    }
    float mx = m;
#pragma unroll
    for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    const float Mn = fmaxf(Mw, mx);
    const float c = Mn == -INFINITY ? 1.0f : exp2f(Mw - Mn);   // rescale what earlier rounds added
    const float f = m == -INFINITY ? 0.0f : exp2f(m - Mn);     // an empty split adds nothing
    float lf = f * l;
#pragma unroll
    for (int off = 16; off; off >>= 1) lf += __shfl_xor_sync(0xFFFFFFFFu, lf, off);
    Lw = Lw * c + lf;
    A.x *= c; A.y *= c; A.z *= c; A.w *= c;
    Mw = Mn;
    const int cnt = min(32, (n - s0 + kW - 1) / kW);
#pragma unroll 8
    for (int j = 0; j < cnt; ++j) {
      const float fj = __shfl_sync(0xFFFFFFFFu, f, j);
      const float4 a = *reinterpret_cast<const float4*>(split_at(s0 + kW * j) + 4 * lane);
      A.x = fmaf(a.x, fj, A.x);
      A.y = fmaf(a.y, fj, A.y);
      A.z = fmaf(a.z, fj, A.z);
      A.w = fmaf(a.w, fj, A.w);
    }
  }
  apart[w][lane] = A;
  if (lane == 0) {
    mpart[w] = Mw;
    lpart[w] = Lw;
  }
  __syncthreads();
  if (w == 0) {
    float M = mpart[0];
#pragma unroll
    for (int k = 1; k < kW; ++k) M = fmaxf(M, mpart[k]);
    float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float Lt = 0.0f;
#pragma unroll
    for (int k = 0; k < kW; ++k) {
      const float g = mpart[k] == -INFINITY ? 0.0f : exp2f(mpart[k] - M);
      const float4 b = apart[k][lane];
      t.x = fmaf(b.x, g, t.x); t.y = fmaf(b.y, g, t.y); t.z = fmaf(b.z, g, t.z); t.w = fmaf(b.w, g, t.w);
      Lt = fmaf(lpart[k], g, Lt);
    }
    const float inv = Lt > 0.0f ? 1.0f / Lt : 0.0f;
    float* o = out + ((size_t)u.b * hq + (size_t)u.kvh * G + h) * kHeadDim + 4 * lane;
    *reinterpret_cast<float4*>(o) = make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
  }
}

template <int G>
cudaError_t launch_g(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units, int n_units,
                     const Split* d_splits, const int32_t* d_cta, int n_ctas, float* d_part, float* out,
                     cudaStream_t s) {
  if (n_ctas > 0) {
    ++P->launches;
    const cudaError_t e = launch_pdl(decode_simt_kernel<G>, dim3((unsigned)n_ctas), dim3(kThreads), 0, s,
                                     (const uint8_t*)P->d_pool, P->int4_offset, (int64_t)P->cfg.n_int2_pages,
                                     P->cfg.num_kv_heads, P->cfg.max_pages_per_request, (const Entry*)P->d_table,
                                     (const __nv_bfloat16*)q, (int)hq, scale_log2, d_units, d_splits, d_cta,
                                     (const int32_t*)P->d_ntab, (const uint32_t*)(P->hdead.empty() ? nullptr : P->d_hdead),
                                     d_part, P->int3_offset, (int64_t)(P->cfg.n_int2_pages + P->cfg.n_int4_pages),
                                     P->fp4_offset,
                                     (int64_t)(P->cfg.n_int2_pages + P->cfg.n_int4_pages + P->cfg.n_int3_pages));
    if (e != cudaSuccess) return e;
  }
  {
    const cudaError_t e = launch_fp_pending(P, q, hq, scale_log2, d_units, d_part, s);
    if (e != cudaSuccess) return e;
  }
  if (P->merge_event) {
    const cudaError_t e = cudaEventRecord(P->merge_event, s);
    if (e != cudaSuccess) return e;
  }
  return launch_merge(P, G, d_units, n_units, d_part, hq, out, s);
}

}  // namespace

cudaError_t launch_merge(kv_pool* P, int g, const Unit* d_units, int n_units, const float* d_part, int hq, float* out,
                         cudaStream_t s) {
  ++P->launches;
  // Programmatic dependent launch: the merge grid is set up while the scan
  // grid drains; its griddepcontrol.wait orders it after the scan's results.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_units * g));
  cfg.blockDim = dim3(256u);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (g) {
    case 1: return cudaLaunchKernelEx(&cfg, merge_kernel<1>, d_units, d_part, hq, out);
    case 2: return cudaLaunchKernelEx(&cfg, merge_kernel<2>, d_units, d_part, hq, out);
    case 3: return cudaLaunchKernelEx(&cfg, merge_kernel<3>, d_units, d_part, hq, out);
    case 4: return cudaLaunchKernelEx(&cfg, merge_kernel<4>, d_units, d_part, hq, out);
    case 5: return cudaLaunchKernelEx(&cfg, merge_kernel<5>, d_units, d_part, hq, out);
    case 6: return cudaLaunchKernelEx(&cfg, merge_kernel<6>, d_units, d_part, hq, out);
    case 7: return cudaLaunchKernelEx(&cfg, merge_kernel<7>, d_units, d_part, hq, out);
    case 8: return cudaLaunchKernelEx(&cfg, merge_kernel<8>, d_units, d_part, hq, out);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_simt(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units,
                               int n_units, const Split* d_splits, const int32_t* d_cta, int n_ctas, float* d_part,
                               float* out, cudaStream_t s) {
  switch (hq / P->cfg.num_kv_heads) {
    case 1: return launch_g<1>(P, q, hq, scale_log2, d_units, n_units, d_splits, d_cta, n_ctas, d_part, out, s);
    case 2: return launch_g<2>(P, q, hq, scale_log2, d_units, n_units, d_splits, d_cta, n_ctas, d_part, out, s);
    case 3: return launch_g<3>(P, q, hq, scale_log2, d_units, n_units, d_splits, d_cta, n_ctas, d_part, out, s);
    case 4: return launch_g<4>(P, q, hq, scale_log2, d_units, n_units, d_splits, d_cta, n_ctas, d_part, out, s);
    case 5: return launch_g<5>(P, q, hq, scale_log2, d_units, n_units, d_splits, d_cta, n_ctas, d_part, out, s);
    case 6: return launch_g<6>(P, q, hq, scale_log2, d_units, n_units, d_splits, d_cta, n_ctas, d_part, out, s);
    case 7: return launch_g<7>(P, q, hq, scale_log2, d_units, n_units, d_splits, d_cta, n_ctas, d_part, out, s);
    case 8: return launch_g<8>(P, q, hq, scale_log2, d_units, n_units, d_splits, d_cta, n_ctas, d_part, out, s);
    default: return cudaErrorInvalidValue;
  }
}

int decode_simt_ctas_per_sm(int g) {
  int n = 0;
  cudaError_t e;
  switch (g) {
    case 1: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<1>, kThreads, 0); break;
    case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<2>, kThreads, 0); break;
    case 4: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<4>, kThreads, 0); break;
    case 8: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<8>, kThreads, 0); break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<4>, kThreads, 0); break;
  }
  return (e == cudaSuccess && n > 0) ? n : 1;
}

}  // namespace kvq
