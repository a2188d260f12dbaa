// Full-precision token lists of the decode (HyQuant, Algorithm 3: after the
// quantized prefix the decode scans the vertical-line tokens, the staging
// buffer and the window, all in full precision, under the same online-softmax
// state; Algorithm 4 FREEZE decides which tokens those are).  Each request has
// one list per kv head, K and V in bf16, laid out [request][kv head][slot][128]
// so that a unit's rows are contiguous.
//
// fp_segment_kernel: persistent warps, one CTA per SM.  Warp gw scans the
// splits [fpw[gw], fpw[gw + 1]): contiguous token ranges of consecutive units
// cut so that every warp gets about the same number of tokens.  Rows stream
// through shared memory in 16-token chunks, two chunks per warp in flight: K
// and V of a chunk are one bulk copy each (a unit's rows are contiguous), and
// chunk c + 2 is issued into the stage of chunk c once c is consumed.  Logits
// are q . k summed in fp32 over exact bf16 x bf16 products; one partial per
// split (acc[128], m, l in the log2 domain), in the format of the page scans,
// so the split merge combines both.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kFpWarps = kFpWarpsPerCta;
constexpr int kFpPartStride = kHeadDim + 4;   // the page scans' partial stride
constexpr int kFpTok = 16;                    // tokens per streamed chunk
constexpr int kRowBytes = kHeadDim * 2;
constexpr int kChunkBytes = kFpTok * kRowBytes;
constexpr uint32_t kFpSpinLimit = 1u << 22;

struct alignas(128) FpWarpSmem {   // bulk copy destinations start on 128-byte boundaries
  uint8_t k[2][kChunkBytes];       // two stages
  uint8_t v[2][kChunkBytes];
  unsigned long long bar[2][2];    // [stage][K, V]
};

template <int G>
constexpr size_t fp_smem_bytes() {
  return kFpWarps * (sizeof(FpWarpSmem) + (size_t)G * kHeadDim * 2 + (size_t)G * kFpTok * 4);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
// acc + lo(a) lo(b) + hi(a) hi(b) for bf16 pairs: exact products, two fp32 roundings
__device__ __forceinline__ float fma2_bf16(uint32_t a, uint32_t b, float acc) {
  asm("{.reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.bf16 %0, al, bl, %0;\n fma.rn.f32.bf16 %0, ah, bh, %0;}"
      : "+f"(acc) : "r"(a), "r"(b));
  return acc;
}

__device__ __forceinline__ void fbar_init(unsigned long long* b) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ void fbulk(void* dst, const void* src, uint32_t bytes, unsigned long long* b) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the buffer was read generically
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(sa(dst)), "l"(src), "r"(bytes), "r"(sa(b)) : "memory");
}
__device__ __forceinline__ bool fbar_wait(unsigned long long* b, uint32_t phase) {
  for (uint32_t it = 0; it < kFpSpinLimit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(sa(b)), "r"(phase) : "memory");
    if (ok) return true;
  }
  return false;
}

// A chunk of the warp's token stream: split, first token, tokens, rows' offset.
struct FpChunk {
  int split, t0, n;
  size_t row;   // index of the chunk's first row in the lists (rows of 128)
};

template <int G>
__global__ void __launch_bounds__(kFpWarps * 32, 1)
    fp_segment_kernel(const uint16_t* __restrict__ q, int hq, float scale_log2, const Unit* __restrict__ units,
                      const Split* __restrict__ fsplits, const int32_t* __restrict__ fpw, int n_fpw, int first_split,
                      const uint16_t* __restrict__ fpk, const uint16_t* __restrict__ fpv, int fp_cap, int hkv,
                      const int32_t* __restrict__ nfp, float* __restrict__ part, uint32_t* __restrict__ status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kFpWarps + w;
  if (gw >= n_fpw) return;   // warps are independent: no block barrier below
  const int sb = fpw[gw], se = fpw[gw + 1];
  if (sb >= se) return;
  FpWarpSmem& S = reinterpret_cast<FpWarpSmem*>(smem)[w];
  uint32_t* qs = reinterpret_cast<uint32_t*>(smem + kFpWarps * sizeof(FpWarpSmem)) + (size_t)w * G * kHeadDim / 2;
  float* ps = reinterpret_cast<float*>(smem + kFpWarps * (sizeof(FpWarpSmem) + (size_t)G * kHeadDim * 2)) +
              (size_t)w * G * kFpTok;
  // token range of a split (its end read at launch when open-ended)
  auto range = [&](int sidx, int& a, int& e) {
    const Split sp = fsplits[sidx];
    const int n_live = nfp[sp.req];
    e = sp.page_end < 0 ? n_live : min(sp.page_end, n_live);
    a = min(sp.page_begin, e);
  };
  // the first chunk at or after token t0 of split sidx, else the first chunk
  // of the next non-empty split; split = se when the stream ends
  auto chunk_at = [&](int sidx, int t0) -> FpChunk {
    int a, e;
    range(sidx, a, e);
    t0 = max(t0, a);
    while (t0 >= e) {
      if (++sidx >= se) return FpChunk{se, 0, 0, 0};
      range(sidx, a, e);
      t0 = a;
    }
    const Unit u = units[fsplits[sidx].unit];
    return FpChunk{sidx, t0, min(kFpTok, e - t0), ((size_t)u.req * hkv + u.kvh) * (size_t)fp_cap + (size_t)t0};
  };
  auto issue = [&](const FpChunk& c, int st) {   // lane 0
    fbulk(S.k[st], fpk + c.row * kHeadDim, (uint32_t)c.n * kRowBytes, &S.bar[st][0]);
    fbulk(S.v[st], fpv + c.row * kHeadDim, (uint32_t)c.n * kRowBytes, &S.bar[st][1]);
  };
  if (lane == 0) {
    fbar_init(&S.bar[0][0]);
    fbar_init(&S.bar[0][1]);
    fbar_init(&S.bar[1][0]);
    fbar_init(&S.bar[1][1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  // chunks c and c + 1 in flight: stage c & 1, barrier phase (c >> 1) & 1
  FpChunk cur = chunk_at(sb, 0);   // the first chunk of split sb (or of a later split; the ones before are empty)
  FpChunk ahead = cur.split < se ? chunk_at(cur.split, cur.t0 + kFpTok) : cur;
  if (lane == 0) {
    if (cur.split < se) issue(cur, 0);
    if (ahead.split < se) issue(ahead, 1);
  }
  uint32_t n_chunk = 0;   // chunks consumed
  const int j = lane & 15, hf = lane >> 4;   // logits: lanes j and j + 16 share token j, 64 channels each
  bool ok = true;
  for (int sidx = sb; sidx < se; ++sidx) {
    const Unit u = units[fsplits[sidx].unit];
    float* out = part + (size_t)(first_split + sidx) * G * kFpPartStride;
    float m[G], lsum[G], acc[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      lsum[h] = 0.0f;
      acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.0f;
    }
    if (cur.split == sidx) {
      // the unit's q rows (bf16 pairs; the scale is applied to the sums)
      __syncwarp();
      const uint32_t* qg = reinterpret_cast<const uint32_t*>(q + ((size_t)u.b * hq + (size_t)u.kvh * G) * kHeadDim);
      for (int x = lane; x < G * kHeadDim / 2; x += 32) qs[x] = qg[x];
      __syncwarp();
    }
    while (cur.split == sidx) {
      const int st = (int)(n_chunk & 1u);
      const uint32_t ph = (n_chunk >> 1) & 1u;
      if (!__all_sync(0xFFFFFFFFu, fbar_wait(&S.bar[st][0], ph))) {
        ok = false;
        break;
      }
      // logits: lane (j, hf) reads 16-byte piece (x + j) mod 8 of its half row
      // at step x, so the 8 lanes of a shared-memory phase hit 8 bank groups
      const bool live = j < cur.n;
      float lg[G];
#pragma unroll
      for (int h = 0; h < G; ++h) lg[h] = 0.0f;
      if (live) {
        const uint8_t* kr = S.k[st] + j * kRowBytes + hf * (kRowBytes / 2);
        const uint32_t* qh = qs + hf * (kHeadDim / 4);
#pragma unroll 2
        for (int x = 0; x < 8; ++x) {
          const int c = (x + j) & 7;
          const uint4 kk = *reinterpret_cast<const uint4*>(kr + 16 * c);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const uint4 qq = *reinterpret_cast<const uint4*>(qh + h * (kHeadDim / 2) + 4 * c);
            float t = lg[h];
            t = fma2_bf16(kk.x, qq.x, t);
            t = fma2_bf16(kk.y, qq.y, t);
            t = fma2_bf16(kk.z, qq.z, t);
            t = fma2_bf16(kk.w, qq.w, t);
            lg[h] = t;
          }
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) lg[h] = (lg[h] + __shfl_xor_sync(0xFFFFFFFFu, lg[h], 16)) * scale_log2;
      // online softmax: the chunk's maximum per head (warp-uniform), the
      // rescale of what earlier chunks added, this chunk's weights
      float corr[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = live ? lg[h] : -INFINITY;
#pragma unroll
        for (int o = 8; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        const float mn = fmaxf(m[h], mx);   // finite: token 0 of the chunk is live
        corr[h] = m[h] == -INFINITY ? 0.0f : exp2f(m[h] - mn);
        m[h] = mn;
        const float p = live ? exp2f(lg[h] - mn) : 0.0f;
        lsum[h] = fmaf(lsum[h], corr[h], hf == 0 ? p : 0.0f);   // per-lane sums, rescaled alike
        if (hf == 0) ps[h * kFpTok + j] = p;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        acc[h][0] *= corr[h];
        acc[h][1] *= corr[h];
        acc[h][2] *= corr[h];
        acc[h][3] *= corr[h];
      }
      if (!__all_sync(0xFFFFFFFFu, fbar_wait(&S.bar[st][1], ph))) {   // also orders ps
        ok = false;
        break;
      }
      // P.V: lane owns channels 4 lane .. 4 lane + 3
      const uint8_t* vr = S.v[st] + 8 * lane;
      int t = 0;
      for (; t + 4 <= cur.n; t += 4) {
        uint2 vv[4];
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) vv[u4] = *reinterpret_cast<const uint2*>(vr + (t + u4) * kRowBytes);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 p4 = *reinterpret_cast<const float4*>(ps + h * kFpTok + t);
          const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
          for (int u4 = 0; u4 < 4; ++u4) {
            acc[h][0] = fmaf(pp[u4], bf_lo(vv[u4].x), acc[h][0]);
            acc[h][1] = fmaf(pp[u4], bf_hi(vv[u4].x), acc[h][1]);
            acc[h][2] = fmaf(pp[u4], bf_lo(vv[u4].y), acc[h][2]);
            acc[h][3] = fmaf(pp[u4], bf_hi(vv[u4].y), acc[h][3]);
          }
        }
      }
      for (; t < cur.n; ++t) {
        const uint2 vv = *reinterpret_cast<const uint2*>(vr + t * kRowBytes);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = ps[h * kFpTok + t];
          acc[h][0] = fmaf(p, bf_lo(vv.x), acc[h][0]);
          acc[h][1] = fmaf(p, bf_hi(vv.x), acc[h][1]);
          acc[h][2] = fmaf(p, bf_lo(vv.y), acc[h][2]);
          acc[h][3] = fmaf(p, bf_hi(vv.y), acc[h][3]);
        }
      }
      __syncwarp();   // stage st and ps read: chunk c + 2 may land in the stage
      const FpChunk nxt = ahead.split < se ? chunk_at(ahead.split, ahead.t0 + kFpTok) : ahead;
      if (nxt.split < se && lane == 0) issue(nxt, st);
      ++n_chunk;
      cur = ahead;
      ahead = nxt;
    }
    if (!ok) break;
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
  if (!ok) {
    if (lane == 0) atomicOr(status, kStatusTimeout);
    // let the copies in flight land (bounded) before the warp leaves: chunks
    // n_chunk and n_chunk + 1 (if issued); the splits not finished read as empty
    const uint32_t c0 = n_chunk, c1 = n_chunk + 1;
    fbar_wait(&S.bar[c0 & 1u][0], (c0 >> 1) & 1u);
    fbar_wait(&S.bar[c0 & 1u][1], (c0 >> 1) & 1u);
    if (ahead.split < se) {
      fbar_wait(&S.bar[c1 & 1u][0], (c1 >> 1) & 1u);
      fbar_wait(&S.bar[c1 & 1u][1], (c1 >> 1) & 1u);
    }
    for (int sidx = max(sb, cur.split); sidx < se; ++sidx)
      for (int h = lane; h < G; h += 32) {
        part[((size_t)(first_split + sidx) * G + h) * kFpPartStride + kHeadDim] = -INFINITY;
        part[((size_t)(first_split + sidx) * G + h) * kFpPartStride + kHeadDim + 1] = 0.0f;
      }
  }
}

// Rows src [n][hkv][128] -> row slot[t] of the lists of request req[t] (one
// per kv head); then the new list lengths (len_req[i] <- len_val[i]).  V = 8:
// 16-byte pieces (both sides 16-byte aligned), V = 1: single elements.
template <int V>
__global__ void fp_store_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                uint16_t* __restrict__ fpk, uint16_t* __restrict__ fpv, int32_t* __restrict__ nfp,
                                const int32_t* __restrict__ req, const int32_t* __restrict__ slot, int64_t n,
                                const int32_t* __restrict__ len_req, const int32_t* __restrict__ len_val, int n_len,
                                int hkv, int fp_cap) {
  constexpr int kPer = kHeadDim / V;   // pieces per row
  const int64_t total = n * hkv * kPer;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total; x += stride) {
    const int64_t row = x / kPer;   // (token, head) in the source order
    const int piece = (int)(x - row * kPer);
    const int64_t t = row / hkv;
    const int h = (int)(row - t * hkv);
    const size_t dst = ((((size_t)req[t] * hkv + h) * fp_cap) + (size_t)slot[t]) * kHeadDim + (size_t)piece * V;
    const size_t src = (size_t)row * kHeadDim + (size_t)piece * V;
    if constexpr (V == 8) {
      *reinterpret_cast<uint4*>(fpk + dst) = *reinterpret_cast<const uint4*>(k + src);
      *reinterpret_cast<uint4*>(fpv + dst) = *reinterpret_cast<const uint4*>(v + src);
    } else {
      fpk[dst] = k[src];
      fpv[dst] = v[src];
    }
  }
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n_len; x += stride) nfp[len_req[x]] = len_val[x];
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

template <int G>
cudaError_t launch_fp_g(kv_pool* P, const uint16_t* q, int32_t hq, float scale_log2, const Unit* d_units,
                        const Split* d_fsplits, const int32_t* d_fpw, int n_fpw, int first_split, float* d_part,
                        cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(fp_segment_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fp_smem_bytes<G>());
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const dim3 grid((unsigned)((n_fpw + kFpWarps - 1) / kFpWarps)), block(kFpWarps * 32);
  fp_segment_kernel<G><<<grid, block, fp_smem_bytes<G>(), s>>>(q, hq, scale_log2, d_units, d_fsplits, d_fpw, n_fpw,
                                                              first_split, P->d_fpk, P->d_fpv, P->fp_cap,
                                                              P->cfg.num_kv_heads, P->d_nfp, d_part, P->d_status);
  return cudaGetLastError();
}

}  // namespace

int fp_workers(const kv_pool* P) { return P->sm_count * kFpWarps; }

cudaError_t launch_fp_segments(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units,
                               const Split* d_fsplits, const int32_t* d_fpw, int n_fpw, int first_split, float* d_part,
                               cudaStream_t s) {
  if (n_fpw <= 0) return cudaSuccess;
  const uint16_t* qq = (const uint16_t*)q;
  cudaError_t e;
#define KVQ_FP_CASE(g)                                                                                          \
  case g:                                                                                                       \
    e = launch_fp_g<g>(P, qq, hq, scale_log2, d_units, d_fsplits, d_fpw, n_fpw, first_split, d_part, s);        \
    break;
  switch (hq / P->cfg.num_kv_heads) {
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
  return e;
}

cudaError_t launch_fp_store(kv_pool* P, const void* k, const void* v, int64_t n, const int32_t* d_req,
                            const int32_t* d_slot, const int32_t* d_len_req, const int32_t* d_len_val, int n_len,
                            cudaStream_t s) {
  const int hkv = P->cfg.num_kv_heads;
  const bool wide = ((uintptr_t)k % 16 == 0) && ((uintptr_t)v % 16 == 0);
  const int64_t work = std::max<int64_t>(n * hkv * (wide ? kHeadDim / 8 : kHeadDim), n_len);
  const int grid = grid_for(work, P->sm_count);
  if (wide)
    fp_store_kernel<8><<<grid, 256, 0, s>>>((const uint16_t*)k, (const uint16_t*)v, P->d_fpk, P->d_fpv, P->d_nfp, d_req,
                                            d_slot, n, d_len_req, d_len_val, n_len, hkv, P->fp_cap);
  else
    fp_store_kernel<1><<<grid, 256, 0, s>>>((const uint16_t*)k, (const uint16_t*)v, P->d_fpk, P->d_fpv, P->d_nfp, d_req,
                                            d_slot, n, d_len_req, d_len_val, n_len, hkv, P->fp_cap);
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
