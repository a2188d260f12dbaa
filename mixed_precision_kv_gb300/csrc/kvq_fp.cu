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
// through shared memory in 16-token chunks, three chunks per warp in flight:
// K and V of a chunk are one bulk copy each (a unit's rows are contiguous),
// and chunk c + 3 is issued into the stage of chunk c once c is consumed.
// Logits and P.V run on the tensor cores (bf16 operands, fp32 accumulation;
// P split into bf16 hi + lo parts); one partial per split (acc[128], m, l in
// the log2 domain), in the format of the page scans, so the split merge
// combines both.
#include <cuda_runtime.h>

#include <atomic>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kFpWarps = kFpWarpsPerCta;
constexpr int kFpPartStride = kHeadDim + 4;   // the page scans' partial stride
constexpr int kFpTok = 16;                    // tokens per streamed chunk
constexpr int kFpStages = 3;                  // chunks in flight per warp
constexpr int kRowBytes = kHeadDim * 2;
constexpr int kChunkBytes = kFpTok * kRowBytes;
constexpr uint32_t kFpSpinLimit = 1u << 22;

struct alignas(128) FpWarpSmem {   // bulk copy destinations start on 128-byte boundaries
  uint8_t k[kFpStages][kChunkBytes];
  uint8_t v[kFpStages][kChunkBytes];
  unsigned long long bar[kFpStages][2];   // [stage][K, V]
  float ps[8][kFpTok];             // P [head][token] of the current chunk
  float corr[8];                   // per-head rescale of the current chunk
};
constexpr size_t kFpSmem = kFpWarps * sizeof(FpWarpSmem);

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(sa(p)) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(sa(p)) : "memory");
}
// d += A B, bf16 operands (exact products), fp32 accumulation
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// two floats as a bf16 pair (round to nearest even): lo -> bits 0..15
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// p = hi + lo with hi = bf16(p), lo = bf16(p - hi): 16 significant bits
__device__ __forceinline__ void split_bf2(float x, float y, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf2(x, y);
  lo = pack_bf2(x - bf_lo(hi), y - bf_hi(hi));
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
__device__ __forceinline__ bool fbar_wait(unsigned long long* b, uint32_t phase, uint32_t limit = kFpSpinLimit) {
  for (uint32_t it = 0; it < limit; ++it) {
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
  int e;        // end of the chunk's split
};

template <int G>
__device__ __forceinline__ void fp_segment_warp(uint8_t* smem, const uint16_t* __restrict__ q, int hq,
                                                float scale_log2, const Unit* __restrict__ units,
                                                const Split* __restrict__ fsplits, const int32_t* __restrict__ fpw,
                                                int n_fpw, int first_split, const uint16_t* __restrict__ fpk,
                                                const uint16_t* __restrict__ fpv, int fp_cap, int hkv,
                                                const int32_t* __restrict__ nfp, float* __restrict__ part,
                                                uint32_t* __restrict__ status, uint32_t first_spins) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kFpWarps + w;
  if (gw >= n_fpw) return;   // warps are independent: no block barrier below
  const int sb = fpw[gw], se = fpw[gw + 1];
  if (sb >= se) return;
  FpWarpSmem& S = reinterpret_cast<FpWarpSmem*>(smem)[w];
  const int r = lane >> 2, i = lane & 3;   // mma fragment coordinates
  const int mi = lane >> 3, mr = lane & 7;   // ldmatrix: the lane addresses row mr of matrix mi
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
      if (++sidx >= se) return FpChunk{se, 0, 0, 0, 0};
      range(sidx, a, e);
      t0 = a;
    }
    const Unit u = units[fsplits[sidx].unit];
    return FpChunk{sidx, t0, min(kFpTok, e - t0), ((size_t)u.req * hkv + u.kvh) * (size_t)fp_cap + (size_t)t0, e};
  };
  // the chunk after c: the next kFpTok tokens of its split without a load,
  // else the first chunk of a later split
  auto chunk_after = [&](const FpChunk& c) -> FpChunk {
    if (c.split >= se) return c;
    const int t0 = c.t0 + kFpTok;
    if (t0 < c.e) return FpChunk{c.split, t0, min(kFpTok, c.e - t0), c.row + kFpTok, c.e};
    return c.split + 1 < se ? chunk_at(c.split + 1, 0) : FpChunk{se, 0, 0, 0, 0};
  };
  auto issue = [&](const FpChunk& c, int st) {   // lane 0
    fbulk(S.k[st], fpk + c.row * kHeadDim, (uint32_t)c.n * kRowBytes, &S.bar[st][0]);
    fbulk(S.v[st], fpv + c.row * kHeadDim, (uint32_t)c.n * kRowBytes, &S.bar[st][1]);
  };
  // rows past a short chunk's end keep earlier chunks' values: start from zeros
  for (int x = lane; x < (int)(2 * kFpStages * kChunkBytes / 16); x += 32)
    reinterpret_cast<uint4*>(&S.k[0][0])[x] = make_uint4(0u, 0u, 0u, 0u);   // k and v are adjacent
  if (lane == 0) {
    for (int st = 0; st < kFpStages; ++st) {
      fbar_init(&S.bar[st][0]);
      fbar_init(&S.bar[st][1]);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  // chunks c .. c + kFpStages - 1 in flight: chunk c in stage c mod kFpStages,
  // barrier phase (c / kFpStages) & 1; ring[x] is chunk c + x
  FpChunk ring[kFpStages];
  ring[0] = chunk_at(sb, 0);   // the first chunk of split sb (or of a later split; the ones before are empty)
#pragma unroll
  for (int x = 1; x < kFpStages; ++x)
    ring[x] = chunk_after(ring[x - 1]);
  if (lane == 0) {
#pragma unroll
    for (int x = 0; x < kFpStages; ++x)
      if (ring[x].split < se) issue(ring[x], x);
  }
  FpChunk& cur = ring[0];
  uint32_t n_chunk = 0;   // chunks consumed
  bool ok = true;
  for (int sidx = sb; sidx < se; ++sidx) {
    const Unit u = units[fsplits[sidx].unit];
    float* out = part + (size_t)(first_split + sidx) * G * kFpPartStride;
    // lane (r, i): softmax state of heads 2i, 2i + 1; O rows r (head r, the
    // hi part of P) and r + 8 (the lo part) of channels 8j + 2i, 8j + 2i + 1
    float m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.0f, 0.0f};
    float acc[16][4];
#pragma unroll
    for (int jt = 0; jt < 16; ++jt) acc[jt][0] = acc[jt][1] = acc[jt][2] = acc[jt][3] = 0.0f;
    // B operand of the logits: column n = head n, k = channel; lane (r, i)
    // holds q[r][16kk + 2i, +1] and q[r][16kk + 2i + 8, +9] (0 past g heads)
    uint32_t qb[8][2];
    {
      const uint32_t* qr = reinterpret_cast<const uint32_t*>(q + ((size_t)u.b * hq + (size_t)u.kvh * G + r) * kHeadDim);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qb[kk][0] = (r < G && cur.split == sidx) ? qr[8 * kk + i] : 0u;
        qb[kk][1] = (r < G && cur.split == sidx) ? qr[8 * kk + i + 4] : 0u;
      }
    }
    while (cur.split == sidx) {
      const int st = (int)(n_chunk % kFpStages);
      const uint32_t ph = (n_chunk / kFpStages) & 1u;
      // the first wait's bound is kFpSpinLimit unless a test shortens it
      if (!__all_sync(0xFFFFFFFFu, fbar_wait(&S.bar[st][0], ph, n_chunk == 0 ? first_spins : kFpSpinLimit))) {
        ok = false;
        break;
      }
      // logits D[token][head] = K q^T on the tensor cores; the list stores
      // 16-byte piece c of row t at piece c ^ (t & 7), so the eight rows of
      // an 8x8 ldmatrix tile sit in eight different bank groups
      const int tk = (mi & 1) * 8 + mr;   // token row this lane addresses
      const int key = (cur.t0 + tk) & 7;
      const uint8_t* krow = S.k[st] + tk * kRowBytes;
      float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a[4];
        ldsm_x4(a, krow + 16 * ((2 * kk + (mi >> 1)) ^ key));
        if (kk & 1) mma_bf16(d1, a[0], a[1], a[2], a[3], qb[kk][0], qb[kk][1]);
        else mma_bf16(d0, a[0], a[1], a[2], a[3], qb[kk][0], qb[kk][1]);
      }
      // online softmax: lane (r, i) holds tokens r, r + 8 of heads 2i, 2i + 1
      const bool va = r < cur.n, vb = r + 8 < cur.n;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float la = (d0[e] + d1[e]) * scale_log2, lb = (d0[2 + e] + d1[2 + e]) * scale_log2;
        float mx = fmaxf(va ? la : -INFINITY, vb ? lb : -INFINITY);
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
        const float mn = fmaxf(m2[e], mx);   // finite: token 0 of the chunk is live
        const float cr = m2[e] == -INFINITY ? 0.0f : exp2f(m2[e] - mn);
        m2[e] = mn;
        const float pa = va ? exp2f(la - mn) : 0.0f, pb = vb ? exp2f(lb - mn) : 0.0f;
        l2[e] = fmaf(l2[e], cr, pa + pb);   // per-lane sums over its two tokens, rescaled alike
        S.ps[2 * i + e][r] = pa;
        S.ps[2 * i + e][r + 8] = pb;
        if (r == 0) S.corr[2 * i + e] = cr;
      }
      __syncwarp();   // K read: the next chunk's K may land; P and the rescale are visible
      if (!__all_sync(0xFFFFFFFFu, fbar_wait(&S.bar[st][1], ph))) {
        ok = false;
        break;
      }
      // P.V on the tensor cores: A = [P_hi; P_lo] (rows r, r + 8: head r),
      // B = V from transposed ldmatrix tiles, 16 channel tiles of 8
      uint32_t a0 = 0u, a1 = 0u, a2 = 0u, a3 = 0u;
      float cr = 1.0f;
      if (r < G) {
        const float2 p01 = *reinterpret_cast<const float2*>(&S.ps[r][2 * i]);
        const float2 p89 = *reinterpret_cast<const float2*>(&S.ps[r][2 * i + 8]);
        split_bf2(p01.x, p01.y, a0, a1);
        split_bf2(p89.x, p89.y, a2, a3);
        cr = S.corr[r];
      }
      if (__any_sync(0xFFFFFFFFu, cr != 1.0f)) {
#pragma unroll
        for (int jt = 0; jt < 16; ++jt) {
          acc[jt][0] *= cr;
          acc[jt][1] *= cr;
          acc[jt][2] *= cr;
          acc[jt][3] *= cr;
        }
      }
      const int tv = (mi & 1) * 8 + mr;
      const int vkey = (cur.t0 + tv) & 7;
      const uint8_t* vrow = S.v[st] + tv * kRowBytes;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        uint32_t b[4];
        ldsm_x4_t(b, vrow + 16 * ((2 * jj + (mi >> 1)) ^ vkey));
        mma_bf16(acc[2 * jj], a0, a1, a2, a3, b[0], b[1]);
        mma_bf16(acc[2 * jj + 1], a0, a1, a2, a3, b[2], b[3]);
      }
      __syncwarp();   // stage st, P and the rescale read: chunk c + kFpStages may land in the stage
      const FpChunk& last = ring[kFpStages - 1];
      const FpChunk nxt = chunk_after(last);
      if (nxt.split < se && lane == 0) issue(nxt, st);
      ++n_chunk;
#pragma unroll
      for (int x = 0; x + 1 < kFpStages; ++x) ring[x] = ring[x + 1];
      ring[kFpStages - 1] = nxt;
    }
    if (!ok) break;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l2[e] += __shfl_xor_sync(0xFFFFFFFFu, l2[e], 4);
      l2[e] += __shfl_xor_sync(0xFFFFFFFFu, l2[e], 8);
      l2[e] += __shfl_xor_sync(0xFFFFFFFFu, l2[e], 16);
    }
    if (r < G) {
#pragma unroll
      for (int jt = 0; jt < 16; ++jt)
        *reinterpret_cast<float2*>(out + r * kFpPartStride + 8 * jt + 2 * i) =
            make_float2(acc[jt][0] + acc[jt][2], acc[jt][1] + acc[jt][3]);
    }
    if (r == 0) {
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (2 * i + e < G) {
          out[(2 * i + e) * kFpPartStride + kHeadDim] = m2[e];
          out[(2 * i + e) * kFpPartStride + kHeadDim + 1] = l2[e];
        }
    }
  }
  if (!ok) {
    if (lane == 0) atomicOr(status, kStatusTimeout);
    // let the copies in flight land (bounded) before the warp leaves: chunks
    // n_chunk .. n_chunk + kFpStages - 1 that were issued; the splits not
    // finished read as empty
    for (int x = 0; x < kFpStages; ++x)
      if (ring[x].split < se) {
        const uint32_t c = n_chunk + (uint32_t)x;
        fbar_wait(&S.bar[c % kFpStages][0], (c / kFpStages) & 1u);
        fbar_wait(&S.bar[c % kFpStages][1], (c / kFpStages) & 1u);
      }
    for (int sidx = max(sb, cur.split); sidx < se; ++sidx)
      for (int h = lane; h < G; h += 32) {
        part[((size_t)(first_split + sidx) * G + h) * kFpPartStride + kHeadDim] = -INFINITY;
        part[((size_t)(first_split + sidx) * G + h) * kFpPartStride + kHeadDim + 1] = 0.0f;
      }
  }
}

// Launched as a programmatic dependent of the page scan: the scan's CTAs
// signal at their start, so these CTAs take SMs as the scan's CTAs retire.
// Everything read here was written before the scan began.  Every thread
// waits for the scan grid before it exits, so that the merge's single wait
// (on this grid) covers both.
template <int G>
__global__ void __launch_bounds__(kFpWarps * 32, 1)
    fp_segment_kernel(const uint16_t* __restrict__ q, int hq, float scale_log2, const Unit* __restrict__ units,
                      const Split* __restrict__ fsplits, const int32_t* __restrict__ fpw, int n_fpw, int first_split,
                      const uint16_t* __restrict__ fpk, const uint16_t* __restrict__ fpv, int fp_cap, int hkv,
                      const int32_t* __restrict__ nfp, float* __restrict__ part, uint32_t* __restrict__ status,
                      uint32_t first_spins) {
  extern __shared__ __align__(128) uint8_t smem[];
  asm volatile("griddepcontrol.launch_dependents;");   // the merge may be staged
  fp_segment_warp<G>(smem, q, hq, scale_log2, units, fsplits, fpw, n_fpw, first_split, fpk, fpv, fp_cap, hkv, nfp,
                     part, status, first_spins);
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Rows src [n][hkv][128] -> row slot[t] of the lists of request req[t] (one
// per kv head); then the new list lengths (len_req[i] <- len_val[i]).  V = 8:
// 16-byte pieces (both sides 16-byte aligned), V = 1: single elements.  A
// list row t keeps its 16-byte piece c at piece c ^ (t & 7).
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
    const int sw = slot[t] & 7;
    const int dpos = V == 8 ? ((piece ^ sw) * 8) : ((((piece >> 3) ^ sw) << 3) | (piece & 7));
    const size_t dst = ((((size_t)req[t] * hkv + h) * fp_cap) + (size_t)slot[t]) * kHeadDim + (size_t)dpos;
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
    // the scratch holds pieces in channel order; the list row (at + t) holds
    // piece c at c ^ ((at + t) & 7)
    uint4* list = reinterpret_cast<uint4*>(which ? fpv : fpk) +
                  ((((size_t)req * hkv + h) * fp_cap) + (size_t)(at + t)) * kPer + (piece ^ ((at + t) & 7));
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
  // function attributes are set once per device (bit = device ordinal)
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!(attr_set.load() >> dev & 1u)) {
    const cudaError_t e =
        cudaFuncSetAttribute(fp_segment_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFpSmem);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(uint64_t(1) << dev);
  }
  const dim3 grid((unsigned)((n_fpw + kFpWarps - 1) / kFpWarps)), block(kFpWarps * 32);
  return launch_pdl(fp_segment_kernel<G>, grid, block, kFpSmem, s, q, hq, scale_log2, d_units, d_fsplits, d_fpw,
                    n_fpw, first_split, (const uint16_t*)P->d_fpk, (const uint16_t*)P->d_fpv, P->fp_cap,
                    P->cfg.num_kv_heads, (const int32_t*)P->d_nfp, d_part, P->d_status,
                    P->first_wait_spins < 0 ? kFpSpinLimit : (uint32_t)P->first_wait_spins);
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

cudaError_t launch_fp_pending(kv_pool* P, const void* q, int32_t hq, float scale_log2, const Unit* d_units,
                              float* d_part, cudaStream_t s) {
  const FpLaunch f = P->fp_pending;
  P->fp_pending = FpLaunch{};
  return launch_fp_segments(P, q, hq, scale_log2, d_units, f.d_fsplits, f.d_fpw, f.n_fpw, f.first_split, d_part, s);
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
